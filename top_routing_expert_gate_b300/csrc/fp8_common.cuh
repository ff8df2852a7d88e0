// Helpers shared by the two E4M3 (FP8) weight kernels (experts_fp8.cu,
// experts_fp8_tm.cu): widening of E4M3 codes to bf16 and the warp-wide
// bounded wait their converter warps use.
#pragma once

#include "tc_common.cuh"

namespace moe {
namespace tc {

// Two E4M3 codes placed in the high bytes of two 16-bit halves ([0, b0, 0, b1])
// -> the two values as bf16x2: sign, exponent and mantissa moved into bf16
// positions with the bias-7 exponent kept, then x 2^120 rebiases to 127
// (subnormal codes are bf16 subnormals before the multiply and come out
// exact).  NaN codes (S.1111.111) are out of contract.
__device__ __forceinline__ uint32_t e4m3x2_hi_to_bf16x2(uint32_t t) {
  const uint32_t bits = (t & 0x80008000u) | ((t >> 4) & 0x07F007F0u);
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(bits), "r"(0x7B807B80u));
  return r;
}

// Byte permute of `a` and zero (selector nibbles 0-3: bytes of a, 4: zero).
__device__ __forceinline__ uint32_t prmt_zero(uint32_t a, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(a), "r"(sel));
  return r;
}

// Four codes (one 32-bit word, code j in byte j) -> bf16x2 of codes 0,1 and 2,3.
__device__ __forceinline__ void e4m3x4_to_bf16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = e4m3x2_hi_to_bf16x2(prmt_zero(w, 0x1404u));
  hi = e4m3x2_hi_to_bf16x2(prmt_zero(w, 0x3424u));
}

// Four codes (one 32-bit word, code j in byte j) -> fp16x2 of codes 0,1 and
// 2,3 with the hardware conversion (every finite E4M3 value is exact in
// fp16, subnormal codes included).
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"((unsigned short)(w & 0xffffu)));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"((unsigned short)(w >> 16)));
}

// Bounded mbarrier wait in every lane; the warp agrees on the outcome.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int* abort,
                                          uint64_t timeout_ns) {
  const bool ok = mbar_wait(bar, parity, abort, timeout_ns);
  return __all_sync(0xffffffffu, ok);
}

}  // namespace tc
}  // namespace moe

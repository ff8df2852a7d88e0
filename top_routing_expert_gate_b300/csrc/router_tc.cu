// Router logits on the 5th-generation tensor cores (tcgen05, sm_103a):
// z = x . W_router^T ("10. 混合专家 MoE：总参数与激活参数", niuwancheng.cn,
// "把一个大 FFN 换成一组小 FFN": the router is a d -> E linear layer).
//
// One 128-token tile per CTA, N = E rounded up to 16 (rows past E read as
// zero), and the reduction over d split across `splits` CTAs when there are
// few token tiles.  Each split writes its own fp32 partial [T, E]; the top-k
// kernel adds the partials in split order, so the logits are deterministic.
//   warp 0      TMA producer: 128x64 x tile + E_pad x 64 W_router tile per
//               k-block (128-byte swizzle) into a ring of as many stages as
//               192 KB holds (4 for 256 experts, 8 for 64 or fewer), so that a
//               small expert count still keeps ~192 KB of loads in flight;
//   warp 1      allocates the accumulator's TMEM columns; one thread issues
//               tcgen05.mma M=128 N=E_pad K=16;
//   warps 2..5  epilogue: tcgen05.ld of its 32 TMEM lanes, stored as row
//               segments through shared memory.
#include "tc_common.cuh"

#include <mutex>

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128;            // tokens per tile
constexpr int BK = 64;             // one 128-byte swizzle span of bf16
constexpr int kMaxStages = 8;
constexpr uint32_t kRingBytes = 192 * 1024;   // the stage ring, whatever the stage size
constexpr uint32_t A_STAGE = BM * BK * 2;   // 16 KB
static_assert(2 * (A_STAGE + kMaxExperts * BK * 2) <= kRingBytes, "two stages of the widest weight tile");
constexpr int kThreads = 192;

struct RouterParams {
  CUtensorMap a_map;   // x [T, d], box 64 x 128
  CUtensorMap b_map;   // W_router [E, d], box 64 x E_pad
  float* partial;      // [splits, T, E]
  int T, E, E_pad, kb_total, kb_per, m_tiles;
  int stages;          // ring depth: as many stages as kRingBytes holds, 2..kMaxStages
  uint32_t tmem_cols;
  int32_t* status;
  uint64_t timeout_ns;
};

constexpr uint32_t kRouterSmemMax = kRingBytes + 256 + 1024;

__global__ void __launch_bounds__(kThreads, 1)
router_gemm_kernel(const __grid_constant__ RouterParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t b_stage = (uint32_t)p.E_pad * 128u;
  const uint32_t sA = base;
  const int STAGES = p.stages;
  const uint32_t sB = base + STAGES * A_STAGE;
  uint8_t* ctrl = smem + STAGES * (A_STAGE + b_stage);
  const uint32_t bar0 = smem_u32(ctrl);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  const uint32_t accf = bar0 + 8u * (2 * STAGES);
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 8 * (2 * STAGES + 2));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 8 * (2 * STAGES + 2) + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = blockIdx.x % p.m_tiles;
  const int split = blockIdx.x / p.m_tiles;
  const int kb0 = split * p.kb_per;
  const int kb1 = min(p.kb_total, kb0 + p.kb_per);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(accf, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  bool failed = false;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns)) {
          failed = true;
          break;
        }
        const uint32_t fb = full_bar(stage);
        mbar_arrive_expect_tx(fb, A_STAGE + b_stage);
        tma_load_2d(sA + stage * A_STAGE, &p.a_map, fb, kb * BK, m * BM);
        tma_load_2d(sB + stage * b_stage, &p.b_map, fb, kb * BK, 0);
        ++issued;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (failed) {
        *abort_flag = 1;
        record_error(p.status, kDevTimeout);
      }
      for (int s = 0; s < STAGES; ++s) {
        if (issued > s) {
          const int armed = (issued - 1 - s) / STAGES + 1;
          mbar_wait(full_bar(s), (uint32_t)((armed - 1) & 1), nullptr, p.timeout_ns);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(BM, (uint32_t)p.E_pad);
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(full_bar(stage), phase, abort_flag, p.timeout_ns)) {
          failed = true;
          break;
        }
        tc_fence_after();
        const uint64_t a_desc = sdesc_k128(sA + stage * A_STAGE);
        const uint64_t b_desc = sdesc_k128(sB + stage * b_stage);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_bf16(tmem_base, a_desc + (uint64_t)(2 * kk), b_desc + (uint64_t)(2 * kk), idesc,
                   (kb > kb0 || kk > 0) ? 1u : 0u);
        mma_commit(empty_bar(stage));
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (failed) {
        *abort_flag = 1;
        record_error(p.status, kDevTimeout);
        mma_commit(drain_bar);
        mbar_wait(drain_bar, 0, nullptr, p.timeout_ns);
      } else {
        mma_commit(accf);
      }
    }
  } else {
    const int q = warp & 3;
    const int t0 = m * BM + q * 32;   // first token of this warp's 32 TMEM lanes
    if (mbar_wait(accf, 0, abort_flag, p.timeout_ns)) {
      tc_fence_after();
      // Every MMA has completed, so the token stages are free: each warp
      // passes its 32 x 16 blocks through a padded tile there, so that a
      // store writes 16 consecutive logits of one token row (two rows per
      // warp instruction) instead of one logit in each of 32 rows.
      float* st = reinterpret_cast<float*>(smem) + q * (32 * 17);
      float* out = p.partial + ((size_t)split * p.T + (size_t)t0) * p.E;
      const int rows = min(32, p.T - t0);
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16);
      for (int c = 0; c < p.E_pad; c += 16) {
        uint32_t v[16];
        tmem_ld_32x32b_x16(tbase + (uint32_t)c, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) st[lane * 17 + j] = bits_f(v[j]);
        __syncwarp();
        const int col = c + (lane & 15);
#pragma unroll 4
        for (int r = lane >> 4; r < rows; r += 2)
          if (col < p.E) out[(size_t)r * p.E + col] = st[r * 17 + (lane & 15)];
        __syncwarp();
      }
    } else if (lane == 0) {
      *abort_flag = 1;
      record_error(p.status, kDevTimeout);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

}  // namespace

RouterPlan plan_router(const moe_config_t& c) {
  RouterPlan r{};
  r.m_tiles = (c.T + BM - 1) / BM;
  r.kb_total = c.d_model / BK;
  int splits = kRouterCtaTarget / (r.m_tiles > 0 ? r.m_tiles : 1);
  if (splits < 1) splits = 1;
  if (splits > kMaxRouterSplits) splits = kMaxRouterSplits;
  if (splits > r.kb_total) splits = r.kb_total;
  r.kb_per = (r.kb_total + splits - 1) / splits;
  r.splits = (r.kb_total + r.kb_per - 1) / r.kb_per;
  return r;
}

cudaError_t launch_router_tc(const moe_config_t& c, const void* x, const void* w_router,
                             float* partial, int32_t* status, cudaStream_t s,
                             LaunchCounter* lc) {
  if (c.T == 0) return cudaSuccess;
  const RouterPlan plan = plan_router(c);
  RouterParams p{};
  p.T = c.T;
  p.E = c.n_experts;
  p.E_pad = (c.n_experts + 15) / 16 * 16;
  p.kb_total = plan.kb_total;
  p.kb_per = plan.kb_per;
  p.m_tiles = plan.m_tiles;
  uint32_t cols = 32;
  while (cols < (uint32_t)p.E_pad) cols <<= 1;
  p.tmem_cols = cols;
  p.partial = partial;
  p.status = status;
  p.timeout_ns = kWaitTimeoutNs;
  if (!make_map(&p.a_map, x, c.d_model, c.T, BM) ||
      !make_map(&p.b_map, w_router, c.d_model, c.n_experts, (uint32_t)p.E_pad))
    return cudaErrorInvalidValue;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(router_gemm_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kRouterSmemMax);
  });
  if (attr_err != cudaSuccess) return attr_err;
  // a few experts make small stages: keep ~192 KB of loads in flight per
  // SM, split among the CTAs an SM must hold for the grid to run in one wave
  const int ctas = plan.m_tiles * plan.splits;
  const int per_sm = (ctas + num_sms() - 1) / num_sms();
  const uint32_t stage_bytes = A_STAGE + (uint32_t)p.E_pad * 128u;
  int stages = (int)(kRingBytes / (uint32_t)per_sm / stage_bytes);
  p.stages = stages < 2 ? 2 : (stages > kMaxStages ? kMaxStages : stages);
  const uint32_t smem = (uint32_t)p.stages * stage_bytes + 256 + 1024;
  router_gemm_kernel<<<ctas, kThreads, smem, s>>>(p);
  count_launch(lc);
  return cudaGetLastError();
}

}  // namespace moe

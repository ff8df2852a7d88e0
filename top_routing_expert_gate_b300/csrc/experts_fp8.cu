// Grouped SwiGLU expert GEMMs with FP8 (E4M3) expert weights on the
// 5th-generation tensor cores (tcgen05, sm_103a).
//
// "10. 混合专家 MoE：总参数与激活参数" (niuwancheng.cn), section
// "推理时：显存按总参数，计算按激活参数": DeepSeek-V3 ships its weights in FP8,
// about one byte per parameter, which halves the bytes a decode step streams.
// A stored weight is an E4M3 code times one fp32 scale per output channel:
//
//   gate/up:  g = s_g * (X W_gate^T),  u = s_u * (X W_up^T),  h = SiLU(g) * u -> bf16
//   down:     Y = s_d * (h W_down^T)                                          -> fp32
//
// with W the E4M3 values.  Every E4M3 value is exact in bf16, so the MMAs
// multiply bf16 x bf16 exactly as in the bf16 kernel and the scales are
// applied once per output in the epilogue.
//
// Same tile layout as experts_tc.cu (tokens in the MMA's M, 128-row token
// tiles, 256 weight rows per tile), with the weight operand widened on chip
// in shared memory.  The weights-in-M kernel of experts_fp8_tm.cu, which
// widens into tensor memory, is faster on both the decode (T = 64) and the
// prefill (T = 8192) DeepSeek-V3-shaped layers; this one serves
// the shapes that kernel does not take (d_model not a multiple of 256, or
// d_ff or d_ff_shared not a multiple of 128).
// Three rings: E4M3 weight tiles (5 slots), bf16 token tiles (3 slots) and
// widened bf16 weight tiles (2 slots):
//   warp 0      TMA producer of the E4M3 weight tiles (256 rows x 64 bytes,
//               unswizzled);
//   warp 1      allocates 512 TMEM columns; one thread issues
//               tcgen05.mma M=128 N=256 K=16 and frees a token slot and a
//               widened slot per k-block;
//   warps 2..5  epilogue (scales, SwiGLU, stores through shared memory);
//   warps 6..13 converters: widen each E4M3 slot into the 128-byte-swizzled
//               bf16 layout the MMA reads (each thread loads its 8 chunks of
//               8 codes before converting any, to keep the loads in flight);
//   warp 14     TMA producer of the 128x64 token tiles.
// E4M3 -> bf16: the byte's sign, exponent and mantissa are moved into bf16
// positions (exponent bias 7 kept), then one bf16x2 multiply by 2^120 rebiases
// to 127; subnormal codes come out exact because the multiply sees them as
// bf16 subnormals.  NaN codes (S.1111.111) are out of contract.
#include "fp8_common.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int QBM = 128;
constexpr int QBK = 64;
constexpr int QBN = 256;
constexpr int QNF = 5;                               // E4M3 weight slots
constexpr int QNA = 3;                               // bf16 token-tile slots
constexpr int QNB = 2;                               // widened bf16 weight slots
constexpr uint32_t QA_STAGE = QBM * QBK * 2;         // 16 KB token tile (bf16)
constexpr uint32_t QB_STAGE = QBN * QBK * 2;         // 32 KB weight tile (bf16, widened)
constexpr uint32_t QF_STAGE = QBN * QBK;             // 16 KB weight tile (E4M3)
constexpr int kQThreads = 480;
constexpr int kConvWarp0 = 6;
constexpr int kConvThreads = 256;                    // warps 6..13
constexpr int kTokWarp = 14;
constexpr uint32_t kQTmemCols = 512;
constexpr int kQMaxGroups = kMaxExperts + 1;
constexpr uint32_t kQCtrlBytes = 256 + 4 * (kQMaxGroups + 1 + 3 * kQMaxGroups);
constexpr uint32_t kQStageWords = 32 * 33;
constexpr uint32_t kQEpiBytes = 4 * kQStageWords * 4;
constexpr uint32_t kQSmemBytes =
    QNF * QF_STAGE + QNA * QA_STAGE + QNB * QB_STAGE + kQEpiBytes + kQCtrlBytes + 1024;
static_assert(kQSmemBytes <= 227 * 1024, "shared memory budget");

enum QMode { kQGateUp = 0, kQDown = 1 };

constexpr int kQBoxes = 4;                           // token boxes of 128, 64, 32, 16 rows

struct QParams {
  CUtensorMap a_map[2][kQBoxes];   // [kind][box]: routed grouped rows / shared-expert rows (bf16)
  CUtensorMap b_map[2];     // E4M3 gate (gate/up) or down weights, box 64 B x 128 / 256 rows
  CUtensorMap u_map[2];     // E4M3 up weights (gate/up only)
  const float* b_scale[2];  // per-row scales of b_map's tensor
  const float* u_scale[2];  // per-row scales of u_map's tensor
  const int32_t* offsets;   // [E + 1]
  void* out[2];
  int ld_out[2];
  int K[2];
  int N[2];
  int b_rows_per_expert;
  int E, T, A;
  int has_shared;
  int32_t* status;
  uint64_t timeout_ns;
};

__device__ __forceinline__ int q_n_tiles(int mode, int N) {
  return mode == kQGateUp ? N / 128 : (N + QBN - 1) / QBN;
}

// Generic-proxy shared-memory writes become visible to the async proxy
// (tensor core operand reads, TMA) once this fence is followed by a barrier.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <int MODE>
__global__ void __launch_bounds__(kQThreads, 1)
grouped_gemm_fp8w_kernel(const __grid_constant__ QParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sB = base;                                   // QNB x 32 KB (1024-aligned)
  const uint32_t sA = sB + QNB * QB_STAGE;                    // QNA x 16 KB
  const uint32_t sF = sA + QNA * QA_STAGE;                    // QNF x 16 KB
  uint8_t* f8 = smem + (sF - base);
  uint8_t* bf = smem;
  uint32_t* epi_stage = reinterpret_cast<uint32_t*>(smem + (sF - base) + QNF * QF_STAGE);
  uint8_t* ctrl = reinterpret_cast<uint8_t*>(epi_stage) + kQEpiBytes;
  const uint32_t bar0 = smem_u32(ctrl);
  // barriers: wfull[QNF], wempty[QNF], afull[QNA], aempty[QNA], full[QNB],
  // empty[QNB], accf[2], acce[2], drain
  constexpr int kNB = 2 * QNF + 2 * QNA + 2 * QNB;
  auto wfull_bar = [&](int s) { return bar0 + 8u * s; };
  auto wempty_bar = [&](int s) { return bar0 + 8u * (QNF + s); };
  auto afull_bar = [&](int s) { return bar0 + 8u * (2 * QNF + s); };
  auto aempty_bar = [&](int s) { return bar0 + 8u * (2 * QNF + QNA + s); };
  auto full_bar = [&](int s) { return bar0 + 8u * (2 * QNF + 2 * QNA + s); };
  auto empty_bar = [&](int s) { return bar0 + 8u * (2 * QNF + 2 * QNA + QNB + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (kNB + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (kNB + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (kNB + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 8 * (kNB + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 8 * (kNB + 5) + 4);
  static_assert(8 * (kNB + 5) + 8 <= 256, "barriers fit the control header");
  int* s_tile_start = reinterpret_cast<int*>(ctrl + 256);
  int* s_row0 = s_tile_start + (kQMaxGroups + 1);
  int* s_rows = s_row0 + kQMaxGroups;
  int* s_mtiles = s_rows + kQMaxGroups;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.E + (p.has_shared ? 1 : 0);
  const int nt_r = q_n_tiles(MODE, p.N[0]);
  const int nt_s = q_n_tiles(MODE, p.N[1]);

  for (int g = threadIdx.x; g < G; g += kQThreads) {
    int r0, rows;
    if (g < p.E) {
      r0 = min(max(p.offsets[g], 0), p.A);
      rows = min(max(p.offsets[g + 1], r0), p.A) - r0;
    } else {
      r0 = 0;
      rows = p.T;
    }
    s_row0[g] = r0;
    s_rows[g] = rows;
    s_mtiles[g] = (rows + QBM - 1) / QBM;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < QNF; ++s) {
      mbar_init(wfull_bar(s), 1);
      mbar_init(wempty_bar(s), kConvThreads / 32);   // one arrival per converter warp
    }
    for (int s = 0; s < QNA; ++s) {
      mbar_init(afull_bar(s), 1);
      mbar_init(aempty_bar(s), 1);
    }
    for (int s = 0; s < QNB; ++s) {
      mbar_init(full_bar(s), kConvThreads / 32);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&p.b_map[0]);
    if (MODE == kQGateUp) prefetch_tensormap(&p.u_map[0]);
  }
  if (warp == kTokWarp && lane == 0) prefetch_tensormap(&p.a_map[0][0]);
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kQTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int s = 0;
    for (int g = 0; g < G; ++g) {
      s_tile_start[g] = s;
      s += s_mtiles[g] * (g < p.E ? nt_r : nt_s);
    }
    s_tile_start[G] = s;
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = s_tile_start[G];

  auto decode = [&](int t, int& g, int& m, int& n) {
    int lo = 0, hi = G;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_tile_start[mid] <= t) lo = mid;
      else hi = mid;
    }
    g = lo;
    const int local = t - s_tile_start[g];
    const int mt = s_mtiles[g];
    n = local / mt;
    m = local - n * mt;
  };

  bool failed = false;
  if (warp == 0) {
    if (lane == 0) {
      // ---------------- E4M3 weight producer ----------------
      int issued = 0;
      for (int t = blockIdx.x; t < total && !failed; t += gridDim.x) {
        int g, m, n;
        decode(t, g, m, n);
        const int kind = g < p.E ? 0 : 1;
        const int nk = p.K[kind] / QBK;
        const int b_row = (kind ? 0 : g * p.b_rows_per_expert) + n * (MODE == kQGateUp ? 128 : QBN);
        for (int kb = 0; kb < nk; ++kb, ++issued) {
          const int fs = issued % QNF;
          const uint32_t fph = (uint32_t)(issued / QNF) & 1u;
          if (!mbar_wait(wempty_bar(fs), fph ^ 1u, abort_flag, p.timeout_ns)) {
            failed = true;
            break;
          }
          const uint32_t fb = wfull_bar(fs);
          mbar_arrive_expect_tx(fb, QF_STAGE);
          const uint32_t dst = sF + fs * QF_STAGE;
          tma_load_2d(dst, &p.b_map[kind], fb, kb * QBK, b_row);
          if (MODE == kQGateUp) tma_load_2d(dst + QF_STAGE / 2, &p.u_map[kind], fb, kb * QBK, b_row);
        }
      }
      if (failed) {
        *abort_flag = 1;
        record_error(p.status, kDevTimeout);
      }
      for (int s = 0; s < QNF; ++s) {
        if (issued > s) {
          const int armed = (issued - 1 - s) / QNF + 1;
          mbar_wait(wfull_bar(s), (uint32_t)((armed - 1) & 1), nullptr, p.timeout_ns);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t idesc = idesc_bf16_f32(QBM, QBN);
      int i = 0, local = 0;
      for (int t = blockIdx.x; t < total && !failed; t += gridDim.x, ++local) {
        int g, m, n;
        decode(t, g, m, n);
        const int kind = g < p.E ? 0 : 1;
        const int nk = p.K[kind] / QBK;
        const int buf = local & 1;
        const uint32_t acc_phase = (uint32_t)(local >> 1) & 1u;
        if (!mbar_wait(acce_bar(buf), acc_phase ^ 1u, abort_flag, p.timeout_ns)) {
          failed = true;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * QBN);
        for (int kb = 0; kb < nk; ++kb, ++i) {
          const int bs = i % QNB, as = i % QNA;
          if (!mbar_wait(afull_bar(as), (uint32_t)(i / QNA) & 1u, abort_flag, p.timeout_ns) ||
              !mbar_wait(full_bar(bs), (uint32_t)(i / QNB) & 1u, abort_flag, p.timeout_ns)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint64_t a_desc = sdesc_k128(sA + as * QA_STAGE);
          const uint64_t b_desc = sdesc_k128(sB + bs * QB_STAGE);
#pragma unroll
          for (int kk = 0; kk < QBK / 16; ++kk)
            mma_bf16(d_tmem, a_desc + (uint64_t)(2 * kk), b_desc + (uint64_t)(2 * kk), idesc,
                     (kb | kk) != 0 ? 1u : 0u);
          mma_commit(aempty_bar(as));
          mma_commit(empty_bar(bs));
        }
        if (failed) break;
        mma_commit(accf_bar(buf));
      }
      if (failed) {
        *abort_flag = 1;
        record_error(p.status, kDevTimeout);
        mma_commit(drain_bar);
        mbar_wait(drain_bar, 0, nullptr, p.timeout_ns);
      }
    }
  } else if (warp == kTokWarp) {
    if (lane == 0) {
      // ---------------- token-tile producer ----------------
      int issued = 0;
      for (int t = blockIdx.x; t < total && !failed; t += gridDim.x) {
        int g, m, n;
        decode(t, g, m, n);
        const int kind = g < p.E ? 0 : 1;
        const int nk = p.K[kind] / QBK;
        const int a_row = s_row0[g] + m * QBM;
        // only the tile's valid rows, rounded up to 16 (decode tiles hold a
        // few rows); rows past them keep stale data and give discarded rows
        const int n_load = (min(QBM, s_rows[g] - m * QBM) + 15) & ~15;
        for (int kb = 0; kb < nk; ++kb, ++issued) {
          const int as = issued % QNA;
          if (!mbar_wait(aempty_bar(as), ((uint32_t)(issued / QNA) & 1u) ^ 1u, abort_flag,
                         p.timeout_ns)) {
            failed = true;
            break;
          }
          mbar_arrive_expect_tx(afull_bar(as), (uint32_t)n_load * (QBK * 2));
          int off = 0;
#pragma unroll
          for (int b = 0; b < kQBoxes; ++b) {
            const int box = 128 >> b;
            while (n_load - off >= box) {
              tma_load_2d(sA + as * QA_STAGE + (uint32_t)off * (QBK * 2), &p.a_map[kind][b],
                          afull_bar(as), kb * QBK, a_row + off);
              off += box;
            }
          }
        }
      }
      if (failed) {
        *abort_flag = 1;
        record_error(p.status, kDevTimeout);
      }
      for (int s = 0; s < QNA; ++s) {
        if (issued > s) {
          const int armed = (issued - 1 - s) / QNA + 1;
          mbar_wait(afull_bar(s), (uint32_t)((armed - 1) & 1), nullptr, p.timeout_ns);
        }
      }
    }
  } else if (warp >= kConvWarp0) {
    // ---------------- converters (warps 6..13) ----------------
    const int ct = threadIdx.x - kConvWarp0 * 32;
    int i = 0;
    for (int t = blockIdx.x; t < total && !failed; t += gridDim.x) {
      int g, m, n;
      decode(t, g, m, n);
      const int kind = g < p.E ? 0 : 1;
      const int nk = p.K[kind] / QBK;
      for (int kb = 0; kb < nk; ++kb, ++i) {
        const int fs = i % QNF, bs = i % QNB;
        if (!warp_wait(empty_bar(bs), ((uint32_t)(i / QNB) & 1u) ^ 1u, abort_flag,
                       p.timeout_ns) ||
            !warp_wait(wfull_bar(fs), (uint32_t)(i / QNF) & 1u, abort_flag, p.timeout_ns)) {
          failed = true;
          break;
        }
        // 256 rows x 8 chunks of 8 codes -> 8 bf16 (16 bytes) at the swizzled
        // chunk; each thread loads its 8 chunks before converting any
        constexpr int kPer = QBN * 8 / kConvThreads;
        const uint8_t* src = f8 + fs * QF_STAGE;
        uint8_t* dst = bf + bs * QB_STAGE;
        uint2 v[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
          const int q = ct + kConvThreads * j;
          v[j] = *reinterpret_cast<const uint2*>(src + (q >> 3) * 64 + (q & 7) * 8);
        }
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
          const int q = ct + kConvThreads * j;
          const int r = q >> 3, c = q & 7;
          uint4 o;
          e4m3x4_to_bf16x4(v[j].x, o.x, o.y);
          e4m3x4_to_bf16x4(v[j].y, o.z, o.w);
          *reinterpret_cast<uint4*>(dst + r * 128 + ((c ^ (r & 7)) << 4)) = o;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(wempty_bar(fs));
          mbar_arrive(full_bar(bs));
        }
      }
    }
    if (failed) {
      *abort_flag = 1;
      if (lane == 0) record_error(p.status, kDevTimeout);
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int q = warp & 3;
    int local = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++local) {
      int g, m, n;
      decode(t, g, m, n);
      const int kind = g < p.E ? 0 : 1;
      const int buf = local & 1;
      const uint32_t acc_phase = (uint32_t)(local >> 1) & 1u;
      if (!mbar_wait(accf_bar(buf), acc_phase, abort_flag, p.timeout_ns)) {
        failed = true;
        break;
      }
      tc_fence_after();
      const int rows_left = s_rows[g] - (m * QBM + q * 32);
      const size_t row_base = (size_t)(kind ? 0 : s_row0[g]) + (size_t)(m * QBM + q * 32);
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * QBN);
      uint32_t* st = epi_stage + q * kQStageWords;
      const size_t srow = (size_t)(kind ? 0 : g * p.b_rows_per_expert);
      if (MODE == kQGateUp) {
        const float* sg = p.b_scale[kind] + srow + (size_t)n * 128;
        const float* su = p.u_scale[kind] + srow + (size_t)n * 128;
        uint32_t* out = reinterpret_cast<uint32_t*>(p.out[kind]);
        const size_t ld2 = (size_t)p.ld_out[kind] / 2;
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
#pragma unroll 1
          for (int hh = 0; hh < 32; hh += 16) {   // 16 columns at a time (registers)
            uint32_t gv[16], uv[16];
            tmem_ld_32x32b_x16(tbase + (uint32_t)(c + hh), gv);
            tmem_ld_32x32b_x16(tbase + 128u + (uint32_t)(c + hh), uv);
            tmem_ld_wait();
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
              const float4 a = __ldg(reinterpret_cast<const float4*>(sg + c + hh) + j4);
              const float4 b = __ldg(reinterpret_cast<const float4*>(su + c + hh) + j4);
              const float h0 = silu_f(bits_f(gv[4 * j4]) * a.x) * (bits_f(uv[4 * j4]) * b.x);
              const float h1 = silu_f(bits_f(gv[4 * j4 + 1]) * a.y) * (bits_f(uv[4 * j4 + 1]) * b.y);
              const float h2 = silu_f(bits_f(gv[4 * j4 + 2]) * a.z) * (bits_f(uv[4 * j4 + 2]) * b.z);
              const float h3 = silu_f(bits_f(gv[4 * j4 + 3]) * a.w) * (bits_f(uv[4 * j4 + 3]) * b.w);
              __nv_bfloat162 p0 = __floats2bfloat162_rn(h0, h1);
              __nv_bfloat162 p1 = __floats2bfloat162_rn(h2, h3);
              st[lane * 33 + hh / 2 + 2 * j4] = *reinterpret_cast<uint32_t*>(&p0);
              st[lane * 33 + hh / 2 + 2 * j4 + 1] = *reinterpret_cast<uint32_t*>(&p1);
            }
          }
          __syncwarp();
          const size_t col2 = ((size_t)n * 128 + (size_t)c) / 2 + (size_t)(lane & 15);
#pragma unroll 4
          for (int r = 0; r < 32; r += 2) {
            const int rr = r + (lane >> 4);
            if (rr < rows_left) out[(row_base + rr) * ld2 + col2] = st[rr * 33 + (lane & 15)];
          }
          __syncwarp();
        }
      } else {
        float* out = reinterpret_cast<float*>(p.out[kind]);
        const size_t ld = (size_t)p.ld_out[kind];
        const int ncols = p.N[kind] - n * QBN;   // > 0, a multiple of 64
        const float* sd = p.b_scale[kind] + srow + (size_t)n * QBN;
#pragma unroll 1
        for (int c = 0; c < QBN; c += 32) {
          if (c >= ncols) break;
#pragma unroll 1
          for (int hh = 0; hh < 32; hh += 16) {
            uint32_t v[16];
            tmem_ld_32x32b_x16(tbase + (uint32_t)(c + hh), v);
            tmem_ld_wait();
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
              const float4 a = __ldg(reinterpret_cast<const float4*>(sd + c + hh) + j4);
              st[lane * 33 + hh + 4 * j4] = __float_as_uint(bits_f(v[4 * j4]) * a.x);
              st[lane * 33 + hh + 4 * j4 + 1] = __float_as_uint(bits_f(v[4 * j4 + 1]) * a.y);
              st[lane * 33 + hh + 4 * j4 + 2] = __float_as_uint(bits_f(v[4 * j4 + 2]) * a.z);
              st[lane * 33 + hh + 4 * j4 + 3] = __float_as_uint(bits_f(v[4 * j4 + 3]) * a.w);
            }
          }
          __syncwarp();
          const size_t col = (size_t)n * QBN + (size_t)c + (size_t)lane;
#pragma unroll 4
          for (int r = 0; r < 32; ++r)
            if (r < rows_left) out[(row_base + r) * ld + col] = bits_f(st[r * 33 + lane]);
          __syncwarp();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce_bar(buf));
    }
    if (failed) {
      *abort_flag = 1;
      if (lane == 0) record_error(p.status, kDevTimeout);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kQTmemCols);
  }
}

template <int MODE>
cudaError_t launch_q(const QParams& p, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(grouped_gemm_fp8w_kernel<MODE>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  grouped_gemm_fp8w_kernel<MODE><<<num_sms(), kQThreads, kQSmemBytes, s>>>(p);
  return cudaGetLastError();
}

// Row-major E4M3 matrix [rows, inner] read in unswizzled boxes of 64 bytes x
// box_rows; rows past the end read as zero.
bool token_maps_q(CUtensorMap (&m)[kQBoxes], const void* ptr, uint64_t inner, uint64_t rows) {
  bool ok = true;
  for (int b = 0; b < kQBoxes; ++b) ok &= make_map(&m[b], ptr, inner, rows, 128u >> b);
  return ok;
}

bool make_map_e4m3(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows,
                   uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {64u, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_gemm_fp8w(const moe_config_t& c, const ExpertArgs& a, int which,
                             cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const int T = c.T, E = c.n_experts, d = c.d_model, F = c.d_ff, Fs = c.d_ff_shared;
  const int A = a.rows > 0 ? a.rows : T * c.top_k;
  const bool has_shared = Fs > 0 && a.ws_gate != nullptr;
  const moe_weight_scales_t& sc = *a.scales;
  QParams p{};
  bool ok = true;
  p.offsets = a.offsets;
  p.E = E;
  p.T = T;
  p.A = A;
  p.has_shared = has_shared ? 1 : 0;
  p.status = a.status;
  p.timeout_ns = kWaitTimeoutNs;
  if (which == kGemmGateUp) {
    ok &= token_maps_q(p.a_map[0], a.x_perm, d, A);
    ok &= token_maps_q(p.a_map[1], a.x, d, T);
    ok &= make_map_e4m3(&p.b_map[0], a.w_gate, d, (uint64_t)E * F, 128);
    ok &= make_map_e4m3(&p.u_map[0], a.w_up, d, (uint64_t)E * F, 128);
    p.b_scale[0] = sc.gate_scale;
    p.u_scale[0] = sc.up_scale;
    if (has_shared) {
      ok &= make_map_e4m3(&p.b_map[1], a.ws_gate, d, Fs, 128);
      ok &= make_map_e4m3(&p.u_map[1], a.ws_up, d, Fs, 128);
      p.b_scale[1] = sc.shared_gate_scale;
      p.u_scale[1] = sc.shared_up_scale;
    } else {
      p.b_map[1] = p.b_map[0];
      p.u_map[1] = p.u_map[0];
      p.b_scale[1] = p.b_scale[0];
      p.u_scale[1] = p.u_scale[0];
    }
    p.out[0] = a.h;
    p.out[1] = a.h_shared;
    p.ld_out[0] = F;
    p.ld_out[1] = Fs;
    p.K[0] = d;
    p.K[1] = d;
    p.N[0] = F;
    p.N[1] = has_shared ? Fs : 128;
    p.b_rows_per_expert = F;
  } else {
    ok &= token_maps_q(p.a_map[0], a.h, F, A);
    ok &= make_map_e4m3(&p.b_map[0], a.w_down, F, (uint64_t)E * d, QBN);
    p.b_scale[0] = sc.down_scale;
    if (has_shared) {
      ok &= token_maps_q(p.a_map[1], a.h_shared, Fs, T);
      ok &= make_map_e4m3(&p.b_map[1], a.ws_down, Fs, d, QBN);
      p.b_scale[1] = sc.shared_down_scale;
    } else {
      for (int b = 0; b < kQBoxes; ++b) p.a_map[1][b] = p.a_map[0][b];
      p.b_map[1] = p.b_map[0];
      p.b_scale[1] = p.b_scale[0];
    }
    p.u_map[0] = p.b_map[0];
    p.u_map[1] = p.b_map[1];
    p.u_scale[0] = p.b_scale[0];
    p.u_scale[1] = p.b_scale[1];
    p.out[0] = a.y_perm;
    p.out[1] = a.y_shared;
    p.ld_out[0] = d;
    p.ld_out[1] = d;
    p.K[0] = F;
    p.K[1] = has_shared ? Fs : F;
    p.N[0] = d;
    p.N[1] = d;
    p.b_rows_per_expert = d;
  }
  if (!ok) return cudaErrorInvalidValue;
  const cudaError_t err = which == kGemmGateUp ? launch_q<kQGateUp>(p, s) : launch_q<kQDown>(p, s);
  count_launch(a.launches);
  return err;
}

}  // namespace moe

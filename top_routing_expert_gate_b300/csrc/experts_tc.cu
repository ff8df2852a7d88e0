// Grouped SwiGLU expert GEMMs on the 5th-generation tensor cores (tcgen05,
// sm_103a): the grouped GEMM that replaces the per-expert loop of the block
// sketch in "10. 混合专家 MoE：总参数与激活参数" (niuwancheng.cn, "把一个大 FFN
// 换成一组小 FFN": tokens routed to the same expert are gathered and
// multiplied in one batch).
//
//   gate/up:  [g | u] = X_e [W_gate,e ; W_up,e]^T,  h = SiLU(g) * u  -> bf16
//   down:     Y_e = h_e W_down,e^T                                   -> fp32
//
// Groups are the E routed experts (rows offsets[e]..offsets[e+1] of the
// grouped activations) plus, when present, the shared expert (all T rows).
// The tile list is derived on the device from `offsets`, so no host
// synchronisation separates dispatch from the GEMMs.
//
// Kernel structure (one persistent CTA per SM, 192 threads):
//   warp 0      TMA producer: 128x64 A tile + 256x64 B tile per k-block
//               (128-byte swizzle) into a 4-stage shared-memory ring;
//   warp 1      allocates 512 TMEM columns; one thread issues
//               tcgen05.mma M=128 N=256 K=16 into one of two 256-column fp32
//               accumulators and commits stage / accumulator barriers;
//   warps 2..5  epilogue: tcgen05.ld of its 32 TMEM lanes, SwiGLU (gate/up)
//               or plain fp32 (down), transposed through shared memory so
//               that each global store writes whole row segments.
// For gate/up, the B tile's first 128 rows are W_gate rows and the next 128
// the matching W_up rows, so one N=256 MMA produces both halves and the
// SwiGLU pairs column j with column 128 + j of the same accumulator.
//
// A group's last token tile is usually partial (an expert of the
// DeepSeek-V3-shaped layer holds ~256 rows, so about one tile in five
// would be mostly padding), and a tokens-in-M MMA costs the same whatever
// rows it holds.  A partial tile therefore runs transposed on the same
// shared-memory stages: two MMAs per K step with the B tile's two 128-row
// weight halves as M and the tile's tokens, rounded up to 16, as N, into
// columns 0.. and 128.. of the accumulator.  Each TMEM lane then holds one
// weight row (gate and up of the same feature in one thread, so the SwiGLU
// still needs no exchange), and the MMA time follows the tile's rows.
#include "tc_common.cuh"

#include <cudaTypedefs.h>

#include <mutex>
#include <stdlib.h>
#include <string.h>

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128;
constexpr int BK = 64;             // one 128-byte swizzle span of bf16
constexpr int BN = 256;            // MMA N (gate/up: 128 gate + 128 up columns)
constexpr int STAGES = 4;
constexpr uint32_t A_STAGE = BM * BK * 2;   // 16 KB
constexpr uint32_t B_STAGE = BN * BK * 2;   // 32 KB
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxGroups = kMaxExperts + 1;
constexpr uint32_t kCtrlBytes = 256 + 4 * (kMaxGroups + 1 + 3 * kMaxGroups);
// Epilogue staging: per epilogue warp, 32 rows x 33 words (one word of
// padding keeps both the row-wise writes and the column-wise reads free of
// bank conflicts).
constexpr uint32_t kStageWords = 32 * 33;
constexpr uint32_t kEpiBytes = 4 * kStageWords * 4;
constexpr uint32_t kSmemBytes = STAGES * (A_STAGE + B_STAGE) + kEpiBytes + kCtrlBytes + 1024;

enum Mode { kGateUp = 0, kDown = 1 };

struct TcParams {
  CUtensorMap a_map[2];   // [0] routed grouped rows, [1] shared-expert rows (128-row box)
  CUtensorMap a_part[2][3];   // the same rows in boxes of 64, 32 and 16 (partial tiles)
  CUtensorMap b_map[2];   // gate (kGateUp) or down (kDown) weights
  CUtensorMap u_map[2];   // up weights (kGateUp only)
  const int32_t* offsets; // [E + 1]
  void* out[2];
  int ld_out[2];          // output row stride, elements
  int K[2];               // reduction length per group kind
  int N[2];               // output columns per group kind
  int b_rows_per_expert;  // rows of one routed expert in b_map[0] / u_map[0]
  int E, T, A;
  int has_shared;
  int32_t* status;
  uint64_t timeout_ns;
  int transpose_partial;  // run a partial token tile transposed (weights in M)
};

__device__ __forceinline__ int n_tiles_of(int mode, int N) {
  return mode == kGateUp ? N / 128 : (N + BN - 1) / BN;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = base + STAGES * A_STAGE;
  uint32_t* epi_stage = reinterpret_cast<uint32_t*>(smem + STAGES * (A_STAGE + B_STAGE));
  uint8_t* ctrl = smem + STAGES * (A_STAGE + B_STAGE) + kEpiBytes;
  const uint32_t bar0 = smem_u32(ctrl);
  // barriers: full[STAGES], empty[STAGES], acc_full[2], acc_empty[2], drain
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 8 * (2 * STAGES + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 8 * (2 * STAGES + 5) + 4);
  int* s_tile_start = reinterpret_cast<int*>(ctrl + 256);
  int* s_row0 = s_tile_start + (kMaxGroups + 1);
  int* s_rows = s_row0 + kMaxGroups;
  int* s_mtiles = s_rows + kMaxGroups;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.E + (p.has_shared ? 1 : 0);
  const int nt_r = n_tiles_of(MODE, p.N[0]);
  const int nt_s = n_tiles_of(MODE, p.N[1]);

  // ---- group table (rows per group, clamped to the grouped buffer) ----
  for (int g = threadIdx.x; g < G; g += kThreads) {
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
    s_mtiles[g] = (rows + BM - 1) / BM;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
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
    prefetch_tensormap(&p.a_map[0]);
    prefetch_tensormap(&p.b_map[0]);
    if (MODE == kGateUp) prefetch_tensormap(&p.u_map[0]);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
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

  // tile t -> (group, m tile, n tile); m varies fastest so CTAs running at
  // the same time share the weight tile (L2 reuse of the B operand).
  auto decode = [&](int t, int& g, int& m, int& n) {
    int lo = 0, hi = G;   // largest g with s_tile_start[g] <= t
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
      // ---------------- TMA producer ----------------
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      for (int t = blockIdx.x; t < total && !failed; t += gridDim.x) {
        int g, m, n;
        decode(t, g, m, n);
        const int kind = g < p.E ? 0 : 1;
        const int nk = p.K[kind] / BK;
        const int a_row = s_row0[g] + m * BM;
        const int b_row = (kind ? 0 : g * p.b_rows_per_expert) + n * (MODE == kGateUp ? 128 : BN);
        // a partial tile run transposed reads only its token rows, rounded
        // up to 16 (the MMA's N)
        const int valid = min(BM, s_rows[g] - m * BM);
        const int n_load = valid < BM && p.transpose_partial ? (valid + 15) & ~15 : BM;
        const uint32_t tx = (uint32_t)n_load * (BK * 2) + B_STAGE;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns)) {
            failed = true;
            break;
          }
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, tx);
          const uint32_t a_dst = sA + stage * A_STAGE;
          const uint32_t b_dst = sB + stage * B_STAGE;
          if (n_load == BM) {
            tma_load_2d(a_dst, &p.a_map[kind], fb, kb * BK, a_row);
          } else {
            // boxes of 64, 32, 16 rows, each starting on a 16-row (2 KB)
            // boundary of the stage, so the swizzle pattern is the full tile's
            int off = 0;
#pragma unroll
            for (int b = 0; b < 3; ++b) {
              const int box = 64 >> b;
              while (n_load - off >= box) {
                tma_load_2d(a_dst + (uint32_t)off * (BK * 2), &p.a_part[kind][b], fb, kb * BK,
                            a_row + off);
                off += box;
              }
            }
          }
          if (MODE == kGateUp) {
            tma_load_2d(b_dst, &p.b_map[kind], fb, kb * BK, b_row);
            tma_load_2d(b_dst + B_STAGE / 2, &p.u_map[kind], fb, kb * BK, b_row);
          } else {
            tma_load_2d(b_dst, &p.b_map[kind], fb, kb * BK, b_row);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (failed) {
        *abort_flag = 1;
        record_error(p.status, kDevTimeout);
      }
      // Never leave with copies in flight: wait (bounded) for the last
      // phase armed on every stage.
      for (int s = 0; s < STAGES; ++s) {
        if (issued > s) {
          const int armed = (issued - 1 - s) / STAGES + 1;
          mbar_wait(full_bar(s), (uint32_t)((armed - 1) & 1), nullptr, p.timeout_ns);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      for (int t = blockIdx.x; t < total && !failed; t += gridDim.x, ++local) {
        int g, m, n;
        decode(t, g, m, n);
        const int kind = g < p.E ? 0 : 1;
        const int nk = p.K[kind] / BK;
        const int buf = local & 1;
        const uint32_t acc_phase = (uint32_t)(local >> 1) & 1u;
        if (!mbar_wait(acce_bar(buf), acc_phase ^ 1u, abort_flag, p.timeout_ns)) {
          failed = true;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
        // a partial token tile runs transposed: weight rows in M, its tokens in N
        const int valid = min(BM, s_rows[g] - m * BM);
        const bool part = valid < BM && p.transpose_partial;
        const uint32_t idesc_t = idesc_bf16_f32(BM, (uint32_t)((valid + 15) & ~15));
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag, p.timeout_ns)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint64_t a_desc = sdesc_k128(sA + stage * A_STAGE);
          const uint64_t b_desc = sdesc_k128(sB + stage * B_STAGE);
          if (!part) {
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              // advance 16 bf16 = 32 bytes along K inside the swizzle span
              mma_bf16(d_tmem, a_desc + (uint64_t)(2 * kk), b_desc + (uint64_t)(2 * kk), idesc,
                       (kb | kk) != 0 ? 1u : 0u);
            }
          } else {
            // D[w, t] for the B tile's two 128-row halves (gate and up
            // weights, or two blocks of 128 down-projection outputs) into
            // columns 0.. and 128.. of the buffer; N = the tokens rounded to 16
            const uint64_t b_desc1 = sdesc_k128(sB + stage * B_STAGE + B_STAGE / 2);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              mma_bf16(d_tmem, b_desc + (uint64_t)(2 * kk), a_desc + (uint64_t)(2 * kk), idesc_t,
                       (kb | kk) != 0 ? 1u : 0u);
              mma_bf16(d_tmem + 128u, b_desc1 + (uint64_t)(2 * kk), a_desc + (uint64_t)(2 * kk),
                       idesc_t, (kb | kk) != 0 ? 1u : 0u);
            }
          }
          mma_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (failed) break;
        mma_commit(accf_bar(buf));
      }
      if (failed) {
        *abort_flag = 1;
        record_error(p.status, kDevTimeout);
        // let every MMA already issued finish before the CTA tears down
        mma_commit(drain_bar);
        mbar_wait(drain_bar, 0, nullptr, p.timeout_ns);
      }
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int q = warp & 3;   // TMEM lane quarter this warp may access
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
      const int valid = min(BM, s_rows[g] - m * BM);   // token rows of the tile
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN);
      if (valid < BM && p.transpose_partial) {
        // Transposed (partial) tile: this thread's TMEM lane is weight row
        // w = 32q + lane of each 128-row half, one column per token.  For a
        // token, the warp's 32 lanes store 32 consecutive outputs.
        const int w = q * 32 + lane;
        const size_t row0 = (size_t)(kind ? 0 : s_row0[g]) + (size_t)(m * BM);
        if (MODE == kGateUp) {
          __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out[kind]) +
                               row0 * p.ld_out[kind] + (size_t)n * 128 + (size_t)w;
#pragma unroll 1
          for (int c0 = 0; c0 < valid; c0 += 16) {
            uint32_t gv[16], uv[16];
            tmem_ld_32x32b_x16(tbase + (uint32_t)c0, gv);
            tmem_ld_32x32b_x16(tbase + 128u + (uint32_t)c0, uv);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (c0 + i < valid)
                out[(size_t)(c0 + i) * p.ld_out[kind]] =
                    __float2bfloat16_rn(silu_f(bits_f(gv[i])) * bits_f(uv[i]));
          }
        } else {
          const int ncols = p.N[kind] - n * BN;   // outputs of this n tile
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            if (half * 128 >= ncols) break;
            const bool fvalid = half * 128 + w < ncols;
            float* out = reinterpret_cast<float*>(p.out[kind]) + row0 * p.ld_out[kind] +
                         (size_t)n * BN + (size_t)(half * 128 + w);
#pragma unroll 1
            for (int c0 = 0; c0 < valid; c0 += 16) {
              uint32_t v[16];
              tmem_ld_32x32b_x16(tbase + (uint32_t)(half * 128 + c0), v);
              tmem_ld_wait();
              if (fvalid) {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  if (c0 + i < valid) out[(size_t)(c0 + i) * p.ld_out[kind]] = bits_f(v[i]);
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce_bar(buf));
        continue;
      }
      // Each thread holds one row of the tile (TMEM lane) for 32 columns per
      // load.  The warp passes its 32 x 32 block through shared memory so
      // that every global store writes contiguous bytes of one or two rows.
      const int rows_left = s_rows[g] - (m * BM + q * 32);   // valid rows of this warp's block
      const size_t row_base = (size_t)(kind ? 0 : s_row0[g]) + (size_t)(m * BM + q * 32);
      uint32_t* st = epi_stage + q * kStageWords;
      if (MODE == kGateUp) {
        uint32_t* out = reinterpret_cast<uint32_t*>(p.out[kind]);   // bf16 pairs
        const size_t ld2 = (size_t)p.ld_out[kind] / 2;
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          uint32_t gv[32], uv[32];
          tmem_ld_32x32b_x32(tbase + (uint32_t)c, gv);
          tmem_ld_32x32b_x32(tbase + 128u + (uint32_t)c, uv);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float h0 = silu_f(bits_f(gv[2 * j])) * bits_f(uv[2 * j]);
            const float h1 = silu_f(bits_f(gv[2 * j + 1])) * bits_f(uv[2 * j + 1]);
            __nv_bfloat162 hv = __floats2bfloat162_rn(h0, h1);
            st[lane * 33 + j] = *reinterpret_cast<uint32_t*>(&hv);
          }
          __syncwarp();
          // two rows of 64 bytes per store: lanes 0..15 row r, lanes 16..31 row r + 1
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
        const int ncols = p.N[kind] - n * BN;   // > 0, a multiple of 64
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          if (c >= ncols) break;
          uint32_t v[32];
          tmem_ld_32x32b_x32(tbase + (uint32_t)c, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) st[lane * 33 + j] = v[j];
          __syncwarp();
          // one row of 128 bytes per store
          const size_t col = (size_t)n * BN + (size_t)c + (size_t)lane;
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
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

template <int MODE>
cudaError_t launch(const TcParams& p, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(grouped_gemm_kernel<MODE>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  grouped_gemm_kernel<MODE><<<num_sms(), kThreads, kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

// Token rows in boxes of 64, 32 and 16 rows, for partial tiles.
bool part_maps(CUtensorMap (&m)[3], const void* ptr, uint64_t inner, uint64_t rows) {
  bool ok = true;
  for (int b = 0; b < 3; ++b) ok &= make_map(&m[b], ptr, inner, rows, 64u >> b);
  return ok;
}

}  // namespace

cudaError_t launch_gemm_tc(const moe_config_t& c, const ExpertArgs& a, int which,
                           cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const int T = c.T, E = c.n_experts, d = c.d_model, F = c.d_ff, Fs = c.d_ff_shared;
  const int A = a.rows > 0 ? a.rows : T * c.top_k;
  const bool has_shared = Fs > 0 && a.ws_gate != nullptr;

  TcParams p1{};
  bool ok = true;
  ok &= make_map(&p1.a_map[0], a.x_perm, d, A, BM);
  ok &= make_map(&p1.a_map[1], a.x, d, T, BM);
  ok &= part_maps(p1.a_part[0], a.x_perm, d, A);
  ok &= part_maps(p1.a_part[1], a.x, d, T);
  ok &= make_map(&p1.b_map[0], a.w_gate, d, (uint64_t)E * F, 128);
  ok &= make_map(&p1.u_map[0], a.w_up, d, (uint64_t)E * F, 128);
  if (has_shared) {
    ok &= make_map(&p1.b_map[1], a.ws_gate, d, Fs, 128);
    ok &= make_map(&p1.u_map[1], a.ws_up, d, Fs, 128);
  } else {
    p1.b_map[1] = p1.b_map[0];
    p1.u_map[1] = p1.u_map[0];
  }
  if (!ok) return cudaErrorInvalidValue;
  p1.offsets = a.offsets;
  p1.out[0] = a.h;
  p1.out[1] = a.h_shared;
  p1.ld_out[0] = F;
  p1.ld_out[1] = Fs;
  p1.K[0] = d;
  p1.K[1] = d;
  p1.N[0] = F;
  p1.N[1] = has_shared ? Fs : 128;
  p1.b_rows_per_expert = F;
  p1.E = E;
  p1.T = T;
  p1.A = A;
  p1.has_shared = has_shared ? 1 : 0;
  p1.status = a.status;
  p1.timeout_ns = kWaitTimeoutNs;
  // a partial token tile runs transposed unless MOE_B300_PARTIAL_TILE=full
  // (a tuning and test override)
  const char* pt = getenv("MOE_B300_PARTIAL_TILE");
  p1.transpose_partial = pt && strcmp(pt, "full") == 0 ? 0 : 1;

  TcParams p2 = p1;
  ok = true;
  ok &= make_map(&p2.a_map[0], a.h, F, A, BM);
  ok &= part_maps(p2.a_part[0], a.h, F, A);
  ok &= make_map(&p2.b_map[0], a.w_down, F, (uint64_t)E * d, BN);
  if (has_shared) {
    ok &= make_map(&p2.a_map[1], a.h_shared, Fs, T, BM);
    ok &= part_maps(p2.a_part[1], a.h_shared, Fs, T);
    ok &= make_map(&p2.b_map[1], a.ws_down, Fs, d, BN);
  } else {
    p2.a_map[1] = p2.a_map[0];
    for (int b = 0; b < 3; ++b) p2.a_part[1][b] = p2.a_part[0][b];
    p2.b_map[1] = p2.b_map[0];
  }
  if (!ok) return cudaErrorInvalidValue;
  p2.u_map[0] = p2.b_map[0];
  p2.u_map[1] = p2.b_map[1];
  p2.out[0] = a.y_perm;
  p2.out[1] = a.y_shared;
  p2.ld_out[0] = d;
  p2.ld_out[1] = d;
  p2.K[0] = F;
  p2.K[1] = has_shared ? Fs : F;
  p2.N[0] = d;
  p2.N[1] = d;
  p2.b_rows_per_expert = d;

  cudaError_t err = which == kGemmGateUp ? launch<kGateUp>(p1, s) : launch<kDown>(p2, s);
  count_launch(a.launches);
  return err;
}

}  // namespace moe

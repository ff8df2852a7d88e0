// Grouped SwiGLU expert GEMMs with the expert weights in the MMA's M
// dimension and the tokens in N (tcgen05, sm_103a).
//
// Same operation as experts_tc.cu, the grouped GEMM that replaces the
// per-expert loop of the block sketch in "10. 混合专家 MoE：总参数与激活参数"
// (niuwancheng.cn, "把一个大 FFN 换成一组小 FFN"):
//
//   gate/up:  h_e = SiLU(X_e W_gate,e^T) * (X_e W_up,e^T)   -> bf16
//   down:     Y_e = h_e W_down,e^T                          -> fp32
//
// computed transposed, D^T = W . X^T: MMA rows (TMEM lanes) are output
// features of one expert and the MMA's N columns are that expert's tokens.
// tcgen05 takes any N that is a multiple of 16 up to 256, so an expert with
// R <= 256 rows is one token tile of round32(R) columns: the padding is below
// 32 rows, where 128-row token tiles waste up to 127 (about a fifth of the
// work when every expert holds ~256 rows, as in the DeepSeek-V3-shaped
// layer).  An expert with 256 < R <= 288 rows is still one token tile: two
// MMAs per K step (N = 256, then the last round32(R) - 256 tokens) into one
// accumulator spanning both halves of tensor memory, so no other pair has to
// stream the same weight tile.  Larger experts are split into
// ceil(R / 256) tiles of round32(R / tiles) columns.
//
// Two CTAs (a cluster pair, on two SMs) share one M = 256 MMA
// (tcgen05 .cta_group::2): each CTA stages its own 128 weight rows and half
// of the tile's tokens, so a pipeline stage costs each CTA 32 KB instead of
// 48 KB and six stages fit in shared memory.
//
// Per CTA (192 threads, one per SM, persistent over pair tiles):
//   warp 0      TMA producer: 128x64 weight tile (gate/up: 64 W_gate rows
//               over the 64 matching W_up rows) + (N/2)x64 token rows per
//               k-block, 128-byte swizzle, 6-stage ring; every copy of both
//               CTAs completes on the even CTA's stage barrier;
//   warp 1      allocates 512 TMEM columns (pair allocation); in the even CTA
//               one thread issues tcgen05.mma.cta_group::2 M=256 N=N K=16
//               into one of two 256-column fp32 accumulators (a tile of more
//               than 256 tokens takes both) and multicasts stage-free /
//               accumulator-full commits to both CTAs;
//   warps 2..5  epilogue on this CTA's 128 lanes (= 128 features, all N
//               tokens).  Gate/up: the warps holding W_gate lanes and those
//               holding the matching W_up lanes swap half of each 32-token
//               chunk through shared memory, then each applies SiLU(g)*u to
//               16 tokens and stores bf16 h; down: every warp stores its fp32
//               features.  They release the accumulator on the even CTA's
//               barrier.
#include "tc_common.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int WM = 128;             // weight rows per CTA (MMA M = 256 per pair)
constexpr int WBK = 64;             // k-block: one 128-byte swizzle span of bf16
constexpr int TN = 256;             // token columns of one MMA (its largest N)
constexpr int TN_BIG = 288;         // token columns of a tile that takes both accumulators
constexpr int TNH = TN_BIG / 2;     // token rows staged by each CTA
constexpr int WSTAGES = 6;
constexpr uint32_t W_STAGE = WM * WBK * 2;    // 16 KB
constexpr uint32_t T_STAGE = TNH * WBK * 2;   // 18 KB: 128 rows of the first MMA + 16 of the second
constexpr uint32_t T_TAIL = (TN / 2) * WBK * 2;   // offset of the second MMA's token rows
constexpr int kWThreads = 192;
constexpr uint32_t kWTmemCols = 512;
constexpr int kWMaxGroups = kMaxExperts + 1;
constexpr uint32_t kXchgBytes = 2 * 32 * 64 * 4;   // two 32-token x 64-feature fp32 buffers
constexpr uint32_t kWCtrlBytes = 256 + 4 * (kWMaxGroups + 1 + 4 * kWMaxGroups);
constexpr uint32_t kWSmemBytes =
    WSTAGES * (W_STAGE + T_STAGE) + kXchgBytes + kWCtrlBytes + 1024;
static_assert(kWSmemBytes <= 227 * 1024, "shared memory budget");

enum WMode { kWGateUp = 0, kWDown = 1 };
constexpr int kTokBoxes = 4;        // token boxes of 128, 64, 32, 16 rows

struct WmParams {
  CUtensorMap w_map[2];             // [kind]: W_gate (box 64 rows) or W_down (box 128 rows)
  CUtensorMap u_map[2];             // [kind]: W_up (box 64 rows), gate/up only
  CUtensorMap t_map[2][kTokBoxes];  // [kind][box]: token rows (x_perm/x or h/h_shared)
  const int32_t* offsets;           // [E + 1]
  void* out[2];                     // h / h_shared (bf16) or y_perm / y_shared (fp32)
  int ld_out[2];                    // output row stride, elements
  int K[2];                         // reduction length per group kind
  int n_feat[2];                    // output features per group kind
  int w_rows_per_expert;            // rows of one routed expert in w_map[0] / u_map[0]
  int E, T, A;
  int has_shared;
  int32_t* status;
  uint64_t timeout_ns;
};

// output features of one pair tile (half of them in each CTA)
__device__ __forceinline__ int feat_per_tile(int mode) { return mode == kWGateUp ? 128 : 2 * WM; }

// Named barrier 1 over the four epilogue warps (128 threads).
__device__ __forceinline__ void epi_bar_sync() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}
// The same barrier, returning to every thread the OR of `v` over the 128.
__device__ __forceinline__ bool epi_bar_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// The two 256-column accumulators in tensor memory, as the MMA issuer and
// the epilogue both walk them over the same tile sequence: a tile of at most
// 256 tokens takes the next buffer in turn, a larger one takes both (columns
// 0..n).  Each buffer counts its uses, which gives the mbarrier phase to wait
// for: the release of its previous use (MMA side) or the completion of its
// current one (epilogue side).
struct AccBuffers {
  int next = 0;
  uint32_t uses0 = 0u, uses1 = 0u;
  __device__ __forceinline__ void take(bool both, int& b0, int& b1) {
    if (both) {
      b0 = 0;
      b1 = 1;
    } else {
      b0 = b1 = next;
      next ^= 1;
    }
  }
  __device__ __forceinline__ uint32_t uses(int b) const { return b ? uses1 : uses0; }
  __device__ __forceinline__ uint32_t free_parity(int b) const { return (uses(b) & 1u) ^ 1u; }
  __device__ __forceinline__ uint32_t full_parity(int b) const { return uses(b) & 1u; }
  // buffers b0..b1 (b0 <= b1) have been used once more
  __device__ __forceinline__ void used(int b0, int b1) {
    if (b0 == 0) ++uses0;
    if (b1 == 1) ++uses1;
  }
};

template <int MODE>
__global__ void __launch_bounds__(kWThreads, 1)
grouped_gemm_wm_kernel(const __grid_constant__ WmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sW = base;
  const uint32_t sT = base + WSTAGES * W_STAGE;
  float* xchg = reinterpret_cast<float*>(smem + WSTAGES * (W_STAGE + T_STAGE));
  uint8_t* ctrl = smem + WSTAGES * (W_STAGE + T_STAGE) + kXchgBytes;
  const uint32_t bar0 = smem_u32(ctrl);
  // barriers: full[WSTAGES], empty[WSTAGES], acc_full[2], acc_empty[2], drain.
  // full and acc_empty are used in the even CTA only.
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (WSTAGES + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * WSTAGES + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * WSTAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * WSTAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 8 * (2 * WSTAGES + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 8 * (2 * WSTAGES + 5) + 4);
  int* s_tile_start = reinterpret_cast<int*>(ctrl + 256);
  int* s_row0 = s_tile_start + (kWMaxGroups + 1);
  int* s_rows = s_row0 + kWMaxGroups;
  int* s_ntok = s_rows + kWMaxGroups;    // token tiles of the group
  int* s_tsize = s_ntok + kWMaxGroups;   // token rows per tile (multiple of 32)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();   // 0: issues the MMAs; 1: its peer
  const int pair = (int)cluster_id_x(), npairs = (int)nclusters_x();
  const int G = p.E + (p.has_shared ? 1 : 0);
  const int fpt = feat_per_tile(MODE);
  const int nf_r = (p.n_feat[0] + fpt - 1) / fpt;
  const int nf_s = (p.n_feat[1] + fpt - 1) / fpt;

  // ---- group table: rows, token tiling (identical in both CTAs) ----
  for (int g = threadIdx.x; g < G; g += kWThreads) {
    int r0, rows;
    if (g < p.E) {
      r0 = min(max(p.offsets[g], 0), p.A);
      rows = min(max(p.offsets[g + 1], r0), p.A) - r0;
    } else {
      r0 = 0;
      rows = p.T;
    }
    int nt = (rows + TN - 1) / TN;
    int ts = 32;
    if (rows > TN && rows <= TN_BIG) {
      nt = 1;                                   // one tile over both accumulators
      ts = (rows + 31) & ~31;                   // <= TN_BIG
    } else if (nt > 0) {
      ts = ((rows + nt - 1) / nt + 31) & ~31;   // <= TN
      nt = (rows + ts - 1) / ts;
    }
    s_row0[g] = r0;
    s_rows[g] = rows;
    s_ntok[g] = nt;
    s_tsize[g] = ts;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < WSTAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 8);   // four epilogue warps in each CTA
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&p.w_map[0]);
    if (MODE == kWGateUp) prefetch_tensormap(&p.u_map[0]);
    prefetch_tensormap(&p.t_map[0][0]);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kWTmemCols);
    tmem_relinquish_pair();
    tc_fence_before();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int s = 0;
    for (int g = 0; g < G; ++g) {
      s_tile_start[g] = s;
      s += s_ntok[g] * (g < p.E ? nf_r : nf_s);
    }
    s_tile_start[G] = s;
  }
  // both CTAs' barriers exist before any copy or commit targets them
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = s_tile_start[G];

  // pair tile t -> (group, feature tile f, token tile j); j varies fastest so
  // the pairs that share a weight tile run at the same time (L2 reuse), and
  // the token tiles of one expert stay in L2 while its feature tiles stream.
  auto decode = [&](int t, int& g, int& f, int& j) {
    int lo = 0, hi = G;   // largest g with s_tile_start[g] <= t
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_tile_start[mid] <= t) lo = mid;
      else hi = mid;
    }
    g = lo;
    const int local = t - s_tile_start[g];
    const int nt = s_ntok[g];
    f = local / nt;
    j = local - f * nt;
  };
  // token rows of tile j of group g, and the MMA N (a multiple of 32) covering them
  auto tile_rows = [&](int g, int j, int& first, int& rows, int& n) {
    const int ts = s_tsize[g];
    first = j * ts;
    rows = min(ts, s_rows[g] - first);
    n = (rows + 31) & ~31;
  };

  bool failed = false;
  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs) ----------------
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      for (int t = pair; t < total && !failed; t += npairs) {
        int g, f, j, first, rows, n;
        decode(t, g, f, j);
        tile_rows(g, j, first, rows, n);
        const int kind = g < p.E ? 0 : 1;
        const int nk = p.K[kind] / WBK;
        // token rows staged by this CTA (multiples of 16): its half of the
        // first MMA's N and, for a tile over 256 tokens, its half of the
        // second MMA's N, staged T_TAIL bytes in
        const int n1 = min(n, TN), n2 = n - n1;
        const int half = n1 >> 1, half2 = n2 >> 1;
        const int w_row = (kind ? 0 : g * p.w_rows_per_expert) + f * fpt + (int)rank * (fpt / 2);
        const int t_row = s_row0[g] + first + (int)rank * half;
        const int t_row2 = s_row0[g] + first + n1 + (int)rank * half2;
        const uint32_t tx_pair = 2u * W_STAGE + (uint32_t)n * (WBK * 2);
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns)) {
            failed = true;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), tx_pair);
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          const uint32_t w_dst = sW + stage * W_STAGE;
          const uint32_t t_dst = sT + stage * T_STAGE;
          tma_load_2d_pair(w_dst, &p.w_map[kind], fb, kb * WBK, w_row);
          if (MODE == kWGateUp)
            tma_load_2d_pair(w_dst + W_STAGE / 2, &p.u_map[kind], fb, kb * WBK, w_row);
          // token rows as boxes of 128, 64, 32, 16; every box starts on a
          // 16-row (2 KB) boundary, so the swizzle pattern is that of one tile
          int off = 0;
#pragma unroll
          for (int b = 0; b < kTokBoxes; ++b) {
            const int box = 128 >> b;
            while (half - off >= box) {
              tma_load_2d_pair(t_dst + (uint32_t)off * (WBK * 2), &p.t_map[kind][b], fb,
                               kb * WBK, t_row + off);
              off += box;
            }
          }
          off = 0;
#pragma unroll
          for (int b = 0; b < kTokBoxes; ++b) {
            const int box = 128 >> b;
            while (half2 - off >= box) {
              tma_load_2d_pair(t_dst + T_TAIL + (uint32_t)off * (WBK * 2), &p.t_map[kind][b],
                               fb, kb * WBK, t_row2 + off);
              off += box;
            }
          }
          ++issued;
          if (++stage == WSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (failed) {
        *abort_flag = 1;
        record_error(p.status, kDevTimeout);
      }
      // Never leave with copies in flight: the even CTA waits (bounded) for
      // the last phase armed on every stage, which counts both CTAs' bytes.
      if (rank == 0) {
        for (int s = 0; s < WSTAGES; ++s) {
          if (issued > s) {
            const int armed = (issued - 1 - s) / WSTAGES + 1;
            mbar_wait_cluster(full_bar(s), (uint32_t)((armed - 1) & 1), nullptr, p.timeout_ns);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (even CTA) ----------------
      int stage = 0;
      uint32_t phase = 0;
      AccBuffers acc;
      for (int t = pair; t < total && !failed; t += npairs) {
        int g, f, j, first, rows, n;
        decode(t, g, f, j);
        tile_rows(g, j, first, rows, n);
        const int kind = g < p.E ? 0 : 1;
        const int nk = p.K[kind] / WBK;
        const int n1 = min(n, TN), n2 = n - n1;
        const uint32_t idesc1 = idesc_bf16_f32(2 * WM, (uint32_t)n1);
        const uint32_t idesc2 = idesc_bf16_f32(2 * WM, (uint32_t)(n2 > 0 ? n2 : 32));
        int b0, b1;
        acc.take(n > TN, b0, b1);
        // wait until the epilogue has released every buffer this tile uses
        for (int b = b0; b <= b1 && !failed; ++b)
          if (!mbar_wait_cluster(acce_bar(b), acc.free_parity(b), abort_flag, p.timeout_ns))
            failed = true;
        if (failed) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(b0 * TN);
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_cluster(full_bar(stage), phase, abort_flag, p.timeout_ns)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint64_t a_desc = sdesc_k128(sW + stage * W_STAGE);
          const uint64_t b_desc = sdesc_k128(sT + stage * T_STAGE);
          const uint64_t b_desc2 = sdesc_k128(sT + stage * T_STAGE + T_TAIL);
#pragma unroll
          for (int kk = 0; kk < WBK / 16; ++kk) {
            // advance 16 bf16 = 32 bytes along K inside the swizzle span
            mma_bf16_pair(d_tmem, a_desc + (uint64_t)(2 * kk), b_desc + (uint64_t)(2 * kk),
                          idesc1, (kb | kk) != 0 ? 1u : 0u);
            if (n2 > 0)
              mma_bf16_pair(d_tmem + (uint32_t)TN, a_desc + (uint64_t)(2 * kk),
                            b_desc2 + (uint64_t)(2 * kk), idesc2, (kb | kk) != 0 ? 1u : 0u);
          }
          mma_commit_pair_mc(empty_bar(stage), 3);
          if (++stage == WSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (failed) break;
        for (int b = b0; b <= b1; ++b) mma_commit_pair_mc(accf_bar(b), 3);
        acc.used(b0, b1);
      }
      if (failed) {
        *abort_flag = 1;
        record_error(p.status, kDevTimeout);
        // let every MMA already issued finish before the pair tears down
        mma_commit_pair(drain_bar);
        mbar_wait(drain_bar, 0, nullptr, p.timeout_ns);
      }
    }
  } else {
    // ---------------- epilogue (warps 2..5, both CTAs) ----------------
    const int q = warp & 3;   // TMEM lane quarter this warp may access
    const uint32_t lead_acce0 = mapa_shared(acce_bar(0), 0);
    const uint32_t lead_acce1 = mapa_shared(acce_bar(1), 0);
    AccBuffers acc;
    uint32_t chunk_no = 0;    // running count of exchange chunks (buffer parity)
    for (int t = pair; t < total; t += npairs) {
      int g, f, j, first, rows, n;
      decode(t, g, f, j);
      tile_rows(g, j, first, rows, n);
      const int kind = g < p.E ? 0 : 1;
      int b0, b1;
      acc.take(n > TN, b0, b1);
      bool ok = true;
      for (int b = b0; b <= b1; ++b)
        ok = ok && mbar_wait_cluster(accf_bar(b), acc.full_parity(b), abort_flag, p.timeout_ns);
      if (MODE == kWGateUp) {
        // the exchange below synchronises the four warps, so all of them
        // must take the same decision on whether to process the tile
        if (epi_bar_any(!ok || *abort_flag != 0)) {
          failed = !ok;
          break;
        }
      } else if (!ok) {
        failed = true;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(b0 * TN);
      const size_t row0 = (size_t)(kind ? 0 : s_row0[g]) + (size_t)first;
      const int feat0 = f * fpt + (int)rank * (fpt / 2);   // this CTA's first feature
      if (MODE == kWGateUp) {
        // lanes 0..63: gate features feat0 + 0..63; lanes 64..127: the same up
        // features.  Per 32-token chunk the gate warps hand their values of
        // tokens 16..31 to the up warps and receive the up values of tokens
        // 0..15, so each of the four warps finishes 16 tokens.
        const bool is_gate = q < 2;
        const int fl = (q & 1) * 32 + lane;   // feature within this CTA's 64
        const int tok0 = is_gate ? 0 : 16;    // tokens of the chunk this warp finishes
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out[kind]) +
                             row0 * p.ld_out[kind] + (size_t)(feat0 + fl);
#pragma unroll 1
        for (int c = 0; c < n; c += 32, ++chunk_no) {
          float* xb = xchg + (chunk_no & 1u) * (32 * 64);
          uint32_t v[32];
          tmem_ld_32x32b_x32(tbase + (uint32_t)c, v);
          tmem_ld_wait();
          // gate values of tokens 16..31 -> xb[1024..); up values of tokens 0..15 -> xb[0..)
#pragma unroll
          for (int i = 0; i < 16; ++i)
            xb[(is_gate ? 1024 : 0) + i * 64 + fl] = bits_f(v[is_gate ? 16 + i : i]);
          epi_bar_sync();
          const int lim = min(16, rows - c - tok0);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            if (i < lim) {
              const float other = xb[(is_gate ? 0 : 1024) + i * 64 + fl];
              const float gv = is_gate ? bits_f(v[i]) : other;
              const float uv = is_gate ? other : bits_f(v[16 + i]);
              out[(size_t)(c + tok0 + i) * p.ld_out[kind]] = __float2bfloat16_rn(silu_f(gv) * uv);
            }
          }
        }
      } else {
        const int feat = feat0 + q * 32 + lane;
        const bool fvalid = feat < p.n_feat[kind];
        float* out = reinterpret_cast<float*>(p.out[kind]) + row0 * p.ld_out[kind] + feat;
#pragma unroll 1
        for (int c = 0; c < n; c += 32) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tbase + (uint32_t)c, v);
          tmem_ld_wait();
          if (fvalid) {
            const int lim = min(32, rows - c);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < lim) out[(size_t)(c + i) * p.ld_out[kind]] = bits_f(v[i]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0)
        for (int b = b0; b <= b1; ++b) mbar_arrive_cluster(b ? lead_acce1 : lead_acce0);
      acc.used(b0, b1);
    }
    if (failed) {
      *abort_flag = 1;
      if (lane == 0) record_error(p.status, kDevTimeout);
    }
  }

  tc_fence_before();
  __syncthreads();
  // neither CTA leaves (or frees tensor memory) while its peer may still
  // read its shared memory or signal its barriers
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kWTmemCols);
  }
}

template <int MODE>
cudaError_t launch_wm(const WmParams& p, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int pairs = 0;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(grouped_gemm_wm_kernel<MODE>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kWSmemBytes);
    if (attr_err != cudaSuccess) return;
    // as many co-resident pairs as the device holds (at most one CTA per SM)
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (num_sms() / 2));
    cfg.blockDim = dim3(kWThreads);
    cfg.dynamicSmemBytes = kWSmemBytes;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_wm_kernel<MODE>, &cfg) != cudaSuccess ||
        n <= 0) {
      (void)cudaGetLastError();
      n = num_sms() / 2;
    }
    pairs = n < num_sms() / 2 ? n : num_sms() / 2;
  });
  if (attr_err != cudaSuccess) return attr_err;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(kWThreads);
  cfg.dynamicSmemBytes = kWSmemBytes;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_wm_kernel<MODE>, p);
}

bool token_maps(CUtensorMap (&m)[kTokBoxes], const void* ptr, uint64_t inner, uint64_t rows) {
  bool ok = true;
  for (int b = 0; b < kTokBoxes; ++b) ok &= make_map(&m[b], ptr, inner, rows, 128u >> b);
  return ok;
}

}  // namespace

cudaError_t launch_gemm_wm(const moe_config_t& c, const ExpertArgs& a, int which,
                           cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const int T = c.T, E = c.n_experts, d = c.d_model, F = c.d_ff, Fs = c.d_ff_shared;
  const int A = a.rows > 0 ? a.rows : T * c.top_k;
  const bool has_shared = Fs > 0 && a.ws_gate != nullptr;

  WmParams p1{};
  bool ok = true;
  ok &= make_map(&p1.w_map[0], a.w_gate, d, (uint64_t)E * F, 64);
  ok &= make_map(&p1.u_map[0], a.w_up, d, (uint64_t)E * F, 64);
  ok &= token_maps(p1.t_map[0], a.x_perm, d, A);
  if (has_shared) {
    ok &= make_map(&p1.w_map[1], a.ws_gate, d, Fs, 64);
    ok &= make_map(&p1.u_map[1], a.ws_up, d, Fs, 64);
    ok &= token_maps(p1.t_map[1], a.x, d, T);
  } else {
    p1.w_map[1] = p1.w_map[0];
    p1.u_map[1] = p1.u_map[0];
    for (int b = 0; b < kTokBoxes; ++b) p1.t_map[1][b] = p1.t_map[0][b];
  }
  if (!ok) return cudaErrorInvalidValue;
  p1.offsets = a.offsets;
  p1.out[0] = a.h;
  p1.out[1] = a.h_shared;
  p1.ld_out[0] = F;
  p1.ld_out[1] = Fs;
  p1.K[0] = d;
  p1.K[1] = d;
  p1.n_feat[0] = F;
  p1.n_feat[1] = has_shared ? Fs : 64;
  p1.w_rows_per_expert = F;
  p1.E = E;
  p1.T = T;
  p1.A = A;
  p1.has_shared = has_shared ? 1 : 0;
  p1.status = a.status;
  p1.timeout_ns = kWaitTimeoutNs;

  WmParams p2 = p1;
  ok = true;
  ok &= make_map(&p2.w_map[0], a.w_down, F, (uint64_t)E * d, WM);
  ok &= token_maps(p2.t_map[0], a.h, F, A);
  if (has_shared) {
    ok &= make_map(&p2.w_map[1], a.ws_down, Fs, d, WM);
    ok &= token_maps(p2.t_map[1], a.h_shared, Fs, T);
  } else {
    p2.w_map[1] = p2.w_map[0];
    for (int b = 0; b < kTokBoxes; ++b) p2.t_map[1][b] = p2.t_map[0][b];
  }
  if (!ok) return cudaErrorInvalidValue;
  p2.u_map[0] = p2.w_map[0];
  p2.u_map[1] = p2.w_map[1];
  p2.out[0] = a.y_perm;
  p2.out[1] = a.y_shared;
  p2.ld_out[0] = d;
  p2.ld_out[1] = d;
  p2.K[0] = F;
  p2.K[1] = has_shared ? Fs : F;
  p2.n_feat[0] = d;
  p2.n_feat[1] = d;
  p2.w_rows_per_expert = d;

  cudaError_t err = which == kGemmGateUp ? launch_wm<kWGateUp>(p1, s) : launch_wm<kWDown>(p2, s);
  count_launch(a.launches);
  return err;
}

}  // namespace moe

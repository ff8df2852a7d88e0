// Grouped SwiGLU expert GEMMs with FP8 (E4M3) expert weights: the weight
// rows are the MMA's M and the widened weight operand lives in tensor memory.
//
// "10. 混合专家 MoE：总参数与激活参数" (niuwancheng.cn), section
// "推理时：显存按总参数，计算按激活参数": DeepSeek-V3 ships its weights in FP8,
// about one byte per parameter, which halves the bytes a decode step streams.
// Same arithmetic as experts_fp8.cu (E4M3 codes widened exactly to bf16,
// bf16 x bf16 -> fp32 MMAs, one fp32 scale per output channel applied to the
// accumulator):
//
//   gate/up:  g = s_g * (X W_gate^T),  u = s_u * (X W_up^T),  h = SiLU(g) * u -> bf16
//   down:     Y = s_d * (h W_down^T)                                          -> fp32
//
// Widening the codes in shared memory (experts_fp8.cu) costs a 2-byte write
// and a 2-byte MMA read per weight on top of the code's own traffic, and
// shared-memory bandwidth then bounds the kernel.  Here the converters write
// the widened weights into tensor memory (tcgen05.st) and tcgen05.mma reads
// its A operand from there; shared memory carries only the codes and the
// token tile.  With the tokens in the MMA's N, a ragged last token tile
// costs MMA time in proportion to its rows (N rounded up to 16).
//
// Tile: 256 weight rows (gate/up: 128 W_gate rows and the same 128 W_up rows;
// down: 256 rows of W_down) x up to TN tokens of one group (TN = 32 or 64 for
// small batches, 128 for prefill; see TmTile), k-blocks of 128.
//   warp 0      TMA producer of the E4M3 weight tiles (2 boxes of 128 rows x
//               128 bytes, 128-byte swizzle) into a 4- to 6-slot ring;
//   warps 1, 3  warp 1 allocates 512 TMEM columns; one thread of each issues,
//               per k-block, the 8 tcgen05.mma (K=16 steps) of its 128-row
//               half: M=128, N = the tile's tokens rounded up to 16, A from
//               tensor memory, B (the tokens) from shared memory;
//   warp 2      TMA producer of the token tiles (valid rows only, rounded up
//               to 16) into a 3- or 2-slot ring;
//   warps 4..7, 16..19  epilogue, two warps per lane quarter: scales,
//               SwiGLU, stores (thread = weight row);
//   warps 8..15 converters: warp (q, half) widens rows 32q..32q+31 of its
//               half into tensor-memory lanes 32q..32q+31, 64 columns (128
//               bf16 of K) per k-block.
// Tensor memory: 128-column widened-A stages (three for 32-token tiles, else
// two; half h at +64h), then the accumulators, 2 x TN columns per buffer
// (half h at +TN·h, one column per token).
//
// fp16 operands (the default): the hardware widens two E4M3 codes to fp16x2
// in one conversion, where bf16 needs a byte permute, shifts, masks and a
// rebiasing multiply per pair, and the widening is what bounds this kernel.
// The MMA then takes fp16 tokens too (A and B of one kind::f16 MMA share a
// type): rows_to_f16 writes each token row (and later each row of h) as
// fp16 * 2^s, with s per row chosen so that the row's largest magnitude lands
// in [2^14, 2^15) - exact for every bf16 value of the row down to 2^-31 of
// its largest - and the epilogue multiplies each token's accumulator by 2^s
// before the weight scale.  Products and sums are then the bf16 path's,
// scaled by powers of two.
#include "fp8_common.cuh"

#include <cuda_fp16.h>

namespace moe {
namespace {

using namespace tc;

constexpr int MBM = 128;                             // weight rows per half
constexpr int MBK = 128;                             // K per k-block (codes per row)
constexpr uint32_t MF_HALF = MBM * MBK;              // 16 KB: 128 rows x 128 codes
constexpr uint32_t MF_STAGE = 2 * MF_HALF;           // 32 KB
constexpr int kMThreads = 640;
constexpr int kMTokWarp = 2;
constexpr int kMMma2Warp = 3;                       // issues the second half's MMAs
constexpr int kMEpiWarp0 = 4;                       // and warps 16..19
constexpr int kMConvWarp0 = 8;
constexpr uint32_t kMTmemCols = 512;
constexpr int kMMaxGroups = kMaxExperts + 1;
constexpr uint32_t kMBarBytes = 512;                 // barriers, TMEM address, abort flag
constexpr uint32_t kMCtrlBytes = kMBarBytes + 4 * (kMMaxGroups + 1 + 3 * kMMaxGroups);
constexpr int kMMaxBoxes = 4;

// Token-tile width TN and what follows from it.  Tensor memory holds kNT
// widened-A stages of 128 columns, then the accumulators (kNAcc buffers of
// 2 x TN columns).
//   TN = 32 (a few tokens per expert, as in decode): three A stages, so the
//     converters run up to three k-blocks ahead of the MMAs, two
//     accumulator buffers, 6 E4M3 and 3 token slots;
//   TN = 64: two A stages, two accumulator buffers (the epilogue of one tile
//     overlaps the next tile's MMAs), 5 E4M3 and 3 token slots;
//   TN = 128 (prefill): two A stages and one 256-column accumulator, so the
//     accumulator is single-buffered; 4 E4M3 and 2 token slots of 32 KB.
template <int TN>
struct TmTile {
  static constexpr int kTN = TN;
  static constexpr int kNT = TN == 32 ? 3 : 2;                    // widened-A stages
  static constexpr int kNF = TN == 32 ? 6 : (TN == 64 ? 5 : 4);   // E4M3 slots
  static constexpr int kNA = TN == 128 ? 2 : 3;                   // token slots
  static constexpr int kNAcc = TN == 128 ? 1 : 2;                 // accumulator buffers
  static constexpr int kBoxes = TN == 32 ? 2 : (TN == 64 ? 3 : 4);   // boxes of TN, TN/2, .., 16 rows
  static constexpr uint32_t kAcc0 = kNT * 128;                    // first accumulator column
  static constexpr uint32_t kASub = TN * 128;        // TN token rows x 64 bf16
  static constexpr uint32_t kAStage = 2 * kASub;     // K = 128
  static constexpr uint32_t kSmem = kNF * MF_STAGE + kNA * kAStage + kMCtrlBytes + 1024;
  static_assert(TN == 32 || TN == 64 || TN == 128, "token tile of 32, 64 or 128 rows");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
  static_assert(kAcc0 + kNAcc * 2 * TN == kMTmemCols, "tensor memory budget");
};

enum MMode { kMGateUp = 0, kMDown = 1 };

struct MParams {
  CUtensorMap a_map[2][kMMaxBoxes];  // [kind][box]: routed grouped rows / shared-expert rows (bf16)
  CUtensorMap b_map[2];     // E4M3 gate (gate/up) or down weights, box 128 B x 128 rows
  CUtensorMap u_map[2];     // E4M3 up weights (gate/up only)
  const float* b_scale[2];  // per-row scales of b_map's tensor
  const float* u_scale[2];  // per-row scales of u_map's tensor
  const int32_t* offsets;   // [E + 1]
  void* out[2];
  int ld_out[2];
  int K[2];
  int N[2];                 // output channels per group (a multiple of 256, gate/up: 128)
  int b_rows_per_expert;
  int E, T, A;
  int has_shared;
  int32_t* status;
  uint64_t timeout_ns;
  // fp16 token rows: the accumulator of token column c of a tile is
  // multiplied by row_scale[kind][r], r being the tile's row (routed rows of
  // gate/up: the token perm[row] / perm_div)
  const float* row_scale[2];
  const int32_t* perm;
  int perm_div;
};

__device__ __forceinline__ int m_n_tiles(int mode, int N) {
  return mode == kMGateUp ? N / 128 : N / 256;
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate);
// A is M rows in M lanes with two bf16 of K per 32-bit column.
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns from registers: thread i writes
// row (lane base + i), columns [col, col + 32).
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

template <int MODE, int TN, bool F16>
__global__ void __launch_bounds__(kMThreads, 1)
grouped_gemm_fp8_tm_kernel(const __grid_constant__ MParams p) {
  using C = TmTile<TN>;
  constexpr int MTN = C::kTN, MNF = C::kNF, MNA = C::kNA, NACC = C::kNAcc, MNT = C::kNT;
  constexpr uint32_t kMAccCol0 = C::kAcc0;
  constexpr uint32_t MA_SUB = C::kASub, MA_STAGE = C::kAStage;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sF = base;                                   // MNF x 32 KB (1024-aligned)
  const uint32_t sA = sF + MNF * MF_STAGE;                    // MNA token slots
  const uint8_t* f8 = smem;
  uint8_t* ctrl = smem + MNF * MF_STAGE + MNA * MA_STAGE;
  const uint32_t bar0 = smem_u32(ctrl);
  // barriers: wfull[MNF], wempty[MNF], afull[MNA], aempty[MNA], tfull[MNT],
  // tempty[MNT], accf[2], acce[2] (NACC used), drain[2]
  constexpr int kNB = 2 * MNF + 2 * MNA + 2 * MNT;
  auto wfull_bar = [&](int s) { return bar0 + 8u * s; };
  auto wempty_bar = [&](int s) { return bar0 + 8u * (MNF + s); };
  auto afull_bar = [&](int s) { return bar0 + 8u * (2 * MNF + s); };
  auto aempty_bar = [&](int s) { return bar0 + 8u * (2 * MNF + MNA + s); };
  auto tfull_bar = [&](int s) { return bar0 + 8u * (2 * MNF + 2 * MNA + s); };
  auto tempty_bar = [&](int s) { return bar0 + 8u * (2 * MNF + 2 * MNA + MNT + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (kNB + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (kNB + 2 + b); };
  auto drain_bar = [&](int h) { return bar0 + 8u * (kNB + 4 + h); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 8 * (kNB + 6));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 8 * (kNB + 6) + 4);
  static_assert(8 * (kNB + 6) + 8 <= kMBarBytes, "barriers fit the control header");
  int* s_tile_start = reinterpret_cast<int*>(ctrl + kMBarBytes);
  int* s_row0 = s_tile_start + (kMMaxGroups + 1);
  int* s_rows = s_row0 + kMMaxGroups;
  int* s_mtiles = s_rows + kMMaxGroups;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.E + (p.has_shared ? 1 : 0);
  const int nt_r = m_n_tiles(MODE, p.N[0]);
  const int nt_s = m_n_tiles(MODE, p.N[1]);

  for (int g = threadIdx.x; g < G; g += kMThreads) {
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
    s_mtiles[g] = (rows + MTN - 1) / MTN;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < MNF; ++s) {
      mbar_init(wfull_bar(s), 1);
      mbar_init(wempty_bar(s), 8);    // one arrival per converter warp
    }
    for (int s = 0; s < MNA; ++s) {
      mbar_init(afull_bar(s), 1);
      mbar_init(aempty_bar(s), 2);    // one commit per MMA issuer
    }
    for (int s = 0; s < MNT; ++s) {
      mbar_init(tfull_bar(s), 8);
      mbar_init(tempty_bar(s), 2);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 2);
      mbar_init(acce_bar(b), 8);      // one arrival per epilogue warp
    }
    mbar_init(drain_bar(0), 1);
    mbar_init(drain_bar(1), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&p.b_map[0]);
    if (MODE == kMGateUp) prefetch_tensormap(&p.u_map[0]);
  }
  if (warp == kMTokWarp && lane == 0) prefetch_tensormap(&p.a_map[0][0]);
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kMTmemCols);
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

  // tile t -> (group, token tile m, weight tile n); m fastest, so the token
  // tiles of one weight tile run together and share it in L2
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
  // tokens of the tile, rounded up to 16 (the MMA's N and the rows loaded)
  auto tile_n = [&](int g, int m) { return (min(MTN, s_rows[g] - m * MTN) + 15) & ~15; };
  // power of two of an fp16 token row (row = grouped row, or token for the shared group)
  auto token_scale = [&](int kind, size_t row) -> float {
    if (MODE == kMGateUp && kind == 0) {
      const int a = __ldg(p.perm + row);
      const int tok = a / p.perm_div;
      row = a < 0 || tok >= p.T ? 0 : (size_t)tok;   // the gather reports a bad row
    }
    return __ldg(p.row_scale[kind] + row);
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
        const int nk = p.K[kind] / MBK;
        const int b_row = (kind ? 0 : g * p.b_rows_per_expert) + n * (MODE == kMGateUp ? 128 : 256);
        for (int kb = 0; kb < nk; ++kb, ++issued) {
          const int fs = issued % MNF;
          const uint32_t fph = (uint32_t)(issued / MNF) & 1u;
          if (!mbar_wait(wempty_bar(fs), fph ^ 1u, abort_flag, p.timeout_ns)) {
            failed = true;
            break;
          }
          const uint32_t fb = wfull_bar(fs);
          mbar_arrive_expect_tx(fb, MF_STAGE);
          const uint32_t dst = sF + fs * MF_STAGE;
          if (MODE == kMGateUp) {
            tma_load_2d(dst, &p.b_map[kind], fb, kb * MBK, b_row);
            tma_load_2d(dst + MF_HALF, &p.u_map[kind], fb, kb * MBK, b_row);
          } else {
            tma_load_2d(dst, &p.b_map[kind], fb, kb * MBK, b_row);
            tma_load_2d(dst + MF_HALF, &p.b_map[kind], fb, kb * MBK, b_row + MBM);
          }
        }
      }
      if (failed) {
        *abort_flag = 1;
        record_error(p.status, kDevTimeout);
      }
      for (int s = 0; s < MNF; ++s) {
        if (issued > s) {
          const int armed = (issued - 1 - s) / MNF + 1;
          mbar_wait(wfull_bar(s), (uint32_t)((armed - 1) & 1), nullptr, p.timeout_ns);
        }
      }
    }
  } else if (warp == 1 || warp == kMMma2Warp) {
    if (lane == 0) {
      // ---------------- MMA issuers: warp 1 the first 128-row half, warp 3
      // the second (each MMA instruction takes its issuing thread tens of
      // cycles, and a small token tile makes sixteen per k-block) ----------
      const int hm = warp == 1 ? 0 : 1;
      int i = 0, local = 0;
      for (int t = blockIdx.x; t < total && !failed; t += gridDim.x, ++local) {
        int g, m, n;
        decode(t, g, m, n);
        const int kind = g < p.E ? 0 : 1;
        const int nk = p.K[kind] / MBK;
        const uint32_t idesc = F16 ? idesc_f16_f32(MBM, (uint32_t)tile_n(g, m))
                                   : idesc_bf16_f32(MBM, (uint32_t)tile_n(g, m));
        const int buf = local % NACC;
        const uint32_t acc_phase = (uint32_t)(local / NACC) & 1u;
        if (!mbar_wait(acce_bar(buf), acc_phase ^ 1u, abort_flag, p.timeout_ns)) {
          failed = true;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + kMAccCol0 + (uint32_t)(buf * 2 * MTN);
        for (int kb = 0; kb < nk; ++kb, ++i) {
          const int as = i % MNA, ts = i % MNT;
          if (!mbar_wait(afull_bar(as), (uint32_t)(i / MNA) & 1u, abort_flag, p.timeout_ns) ||
              !mbar_wait(tfull_bar(ts), (uint32_t)(i / MNT) & 1u, abort_flag, p.timeout_ns)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint32_t a_tmem = tmem_base + (uint32_t)(ts * 128);
#pragma unroll
          for (int kk = 0; kk < MBK / 16; ++kk) {
            const uint64_t b_desc =
                sdesc_k128(sA + as * MA_STAGE + (uint32_t)(kk >> 2) * MA_SUB) +
                (uint64_t)(2 * (kk & 3));
            const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
            mma_bf16_ta(d_tmem + (uint32_t)(hm * MTN), a_tmem + (uint32_t)(hm * 64 + 8 * kk),
                        b_desc, idesc, acc);
          }
          mma_commit(aempty_bar(as));
          mma_commit(tempty_bar(ts));
        }
        if (failed) break;
        mma_commit(accf_bar(buf));
      }
      if (failed) {
        *abort_flag = 1;
        record_error(p.status, kDevTimeout);
        mma_commit(drain_bar(hm));
        mbar_wait(drain_bar(hm), 0, nullptr, p.timeout_ns);
      }
    }
  } else if (warp == kMTokWarp) {
    if (lane == 0) {
      // ---------------- token-tile producer ----------------
      int issued = 0;
      for (int t = blockIdx.x; t < total && !failed; t += gridDim.x) {
        int g, m, n;
        decode(t, g, m, n);
        const int kind = g < p.E ? 0 : 1;
        const int nk = p.K[kind] / MBK;
        const int a_row = s_row0[g] + m * MTN;
        // rows between the valid ones and the rounded count belong to the
        // next group or lie past the buffer (zero-filled); their output
        // columns are discarded
        const int n_load = tile_n(g, m);
        for (int kb = 0; kb < nk; ++kb, ++issued) {
          const int as = issued % MNA;
          if (!mbar_wait(aempty_bar(as), ((uint32_t)(issued / MNA) & 1u) ^ 1u, abort_flag,
                         p.timeout_ns)) {
            failed = true;
            break;
          }
          mbar_arrive_expect_tx(afull_bar(as), (uint32_t)n_load * 256u);
#pragma unroll
          for (int sub = 0; sub < 2; ++sub) {
            int off = 0;
#pragma unroll
            for (int b = 0; b < C::kBoxes; ++b) {
              const int box = MTN >> b;
              while (n_load - off >= box) {
                tma_load_2d(sA + as * MA_STAGE + (uint32_t)sub * MA_SUB + (uint32_t)off * 128u,
                            &p.a_map[kind][b], afull_bar(as), kb * MBK + 64 * sub, a_row + off);
                off += box;
              }
            }
          }
        }
      }
      if (failed) {
        *abort_flag = 1;
        record_error(p.status, kDevTimeout);
      }
      for (int s = 0; s < MNA; ++s) {
        if (issued > s) {
          const int armed = (issued - 1 - s) / MNA + 1;
          mbar_wait(afull_bar(s), (uint32_t)((armed - 1) & 1), nullptr, p.timeout_ns);
        }
      }
    }
  } else if (warp >= kMConvWarp0 && warp < kMConvWarp0 + 8) {
    // ---------------- converters (warps 8..15) ----------------
    const int q = warp & 3;                    // tensor-memory lane quarter
    const int half = (warp - kMConvWarp0) >> 2;
    const int r = q * 32 + lane;               // weight row within the half
    const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(half * 64);
    int i = 0;
    for (int t = blockIdx.x; t < total && !failed; t += gridDim.x) {
      int g, m, n;
      decode(t, g, m, n);
      const int kind = g < p.E ? 0 : 1;
      const int nk = p.K[kind] / MBK;
      for (int kb = 0; kb < nk; ++kb, ++i) {
        const int fs = i % MNF, ts = i % MNT;
        if (!warp_wait(tempty_bar(ts), ((uint32_t)(i / MNT) & 1u) ^ 1u, abort_flag,
                           p.timeout_ns) ||
            !warp_wait(wfull_bar(fs), (uint32_t)(i / MNF) & 1u, abort_flag, p.timeout_ns)) {
          failed = true;
          break;
        }
        tc_fence_after();
        // row r: 8 chunks of 16 codes; chunk c sits at chunk c ^ (r & 7) (the
        // 128-byte swizzle), which also spreads a warp's loads over all banks
        const uint8_t* row = f8 + fs * MF_STAGE + half * MF_HALF + r * MBK;
        uint4 v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c)
          v[c] = *reinterpret_cast<const uint4*>(row + ((c ^ (r & 7)) << 4));
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t o[32];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 w = v[4 * h2 + c];
            if (F16) {
              e4m3x4_to_f16x4(w.x, o[8 * c + 0], o[8 * c + 1]);
              e4m3x4_to_f16x4(w.y, o[8 * c + 2], o[8 * c + 3]);
              e4m3x4_to_f16x4(w.z, o[8 * c + 4], o[8 * c + 5]);
              e4m3x4_to_f16x4(w.w, o[8 * c + 6], o[8 * c + 7]);
            } else {
              e4m3x4_to_bf16x4(w.x, o[8 * c + 0], o[8 * c + 1]);
              e4m3x4_to_bf16x4(w.y, o[8 * c + 2], o[8 * c + 3]);
              e4m3x4_to_bf16x4(w.z, o[8 * c + 4], o[8 * c + 5]);
              e4m3x4_to_bf16x4(w.w, o[8 * c + 6], o[8 * c + 7]);
            }
          }
          tmem_st_32x32b_x32(t_row + (uint32_t)(ts * 128 + 32 * h2), o);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(wempty_bar(fs));
          mbar_arrive(tfull_bar(ts));
        }
      }
    }
    if (failed) {
      *abort_flag = 1;
      if (lane == 0) record_error(p.status, kDevTimeout);
    }
  } else if (warp >= kMEpiWarp0) {
    // ---------------- epilogue (warps 4..7 and 16..19) ----------------
    // two warps per lane quarter: part 0 (warps 4..7) and part 1 (16..19)
    // split the tile's columns (gate/up) or its two 128-row halves (down)
    const int q = warp & 3;
    const int part = warp >= 16 ? 1 : 0;
    const int f = q * 32 + lane;               // weight row within a half
    int local = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++local) {
      int g, m, n;
      decode(t, g, m, n);
      const int kind = g < p.E ? 0 : 1;
      const int buf = local % NACC;
      const uint32_t acc_phase = (uint32_t)(local / NACC) & 1u;
      if (!mbar_wait(accf_bar(buf), acc_phase, abort_flag, p.timeout_ns)) {
        failed = true;
        break;
      }
      tc_fence_after();
      const int n_valid = min(MTN, s_rows[g] - m * MTN);
      const size_t row_base = (size_t)(kind ? 0 : s_row0[g]) + (size_t)(m * MTN);
      const uint32_t tacc =
          tmem_base + ((uint32_t)(q * 32) << 16) + kMAccCol0 + (uint32_t)(buf * 2 * MTN);
      const size_t srow = (size_t)(kind ? 0 : g * p.b_rows_per_expert);
      const size_t ld = (size_t)p.ld_out[kind];
      if (MODE == kMGateUp) {
        const size_t col = (size_t)n * 128 + (size_t)f;
        const float sg = __ldg(p.b_scale[kind] + srow + col);
        const float su = __ldg(p.u_scale[kind] + srow + col);
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out[kind]);
        const int lo = part * (MTN / 2), hi = min(n_valid, lo + MTN / 2);
#pragma unroll 1
        for (int c0 = lo; c0 < hi; c0 += 16) {
          // the 16 tokens' row scales: lane i fetches token c0 + (i & 15)'s,
          // then each is broadcast from its lane
          float rs_lane = 1.f;
          if (F16 && c0 + (lane & 15) < hi)
            rs_lane = token_scale(kind, row_base + (size_t)(c0 + (lane & 15)));
          uint32_t gv[16], uv[16];
          tmem_ld_32x32b_x16(tacc + (uint32_t)c0, gv);
          tmem_ld_32x32b_x16(tacc + (uint32_t)(MTN + c0), uv);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float rs = F16 ? __shfl_sync(0xffffffffu, rs_lane, j) : 1.f;
            if (c0 + j < hi) {
              float gj = bits_f(gv[j]), uj = bits_f(uv[j]);
              if (F16) {
                gj *= rs;
                uj *= rs;
              }
              const float hv = silu_f(gj * sg) * (uj * su);
              out[(row_base + (size_t)(c0 + j)) * ld + col] = __float2bfloat16_rn(hv);
            }
          }
        }
      } else {
        float* out = reinterpret_cast<float*>(p.out[kind]);
        {
          const int hf = part;
          const size_t col = (size_t)n * 256 + (size_t)(hf * 128 + f);
          const float sd = __ldg(p.b_scale[kind] + srow + col);
#pragma unroll 1
          for (int c0 = 0; c0 < n_valid; c0 += 16) {
            float rs_lane = 1.f;
            if (F16 && c0 + (lane & 15) < n_valid)
              rs_lane = token_scale(kind, row_base + (size_t)(c0 + (lane & 15)));
            uint32_t v[16];
            tmem_ld_32x32b_x16(tacc + (uint32_t)(hf * MTN + c0), v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float rs = F16 ? __shfl_sync(0xffffffffu, rs_lane, j) : 1.f;
              if (c0 + j < n_valid) {
                float vj = bits_f(v[j]);
                if (F16) vj *= rs;
                out[(row_base + (size_t)(c0 + j)) * ld + col] = vj * sd;
              }
            }
          }
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
    tmem_dealloc(tmem_base, kMTmemCols);
  }
}

template <int MODE, int TN, bool F16>
cudaError_t launch_m(const MParams& p, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(grouped_gemm_fp8_tm_kernel<MODE, TN, F16>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    TmTile<TN>::kSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  grouped_gemm_fp8_tm_kernel<MODE, TN, F16><<<num_sms(), kMThreads, TmTile<TN>::kSmem, s>>>(p);
  return cudaGetLastError();
}

// Row r of `in` (bf16, vec 8-element vectors per row) -> `out` (fp16, may be
// `in` itself) as in[r] * 2^-s with s = clamp(floor(log2 max|in[r]|) - 14,
// -126, 113), so the row's largest magnitude lands in [2^14, 2^15);
// scale[r] = 2^s.  One warp per row: the maximum first, then the rewrite.
__global__ void __launch_bounds__(256)
rows_to_f16_kernel(const uint4* in, uint4* out, float* __restrict__ scale, int rows, int vec) {
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  for (int r = blockIdx.x * warps + (threadIdx.x >> 5); r < rows; r += gridDim.x * warps) {
    const uint4* src = in + (size_t)r * vec;
    uint32_t mx = 0;   // bf16 magnitudes compare as integers
    for (int v = lane; v < vec; v += 32) {
      const uint4 u = src[v];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) mx = max(mx, max(w[i] & 0x7fffu, (w[i] >> 16) & 0x7fffu));
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    const int s = mx == 0 ? 0 : min(max((int)(mx >> 7) - 127 - 14, -126), 113);
    const float down = __int_as_float((127 - s) << 23);   // 2^-s
    uint4* dst = out + (size_t)r * vec;
    for (int v = lane; v < vec; v += 32) {
      const uint4 u = src[v];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float lo = __uint_as_float(w[i] << 16) * down;
        const float hi = __uint_as_float(w[i] & 0xffff0000u) * down;
        __half2 h = __floats2half2_rn(lo, hi);
        o[i] = *reinterpret_cast<uint32_t*>(&h);
      }
      dst[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (lane == 0) scale[r] = __int_as_float((127 + s) << 23);
  }
}

// Token boxes of tn, tn/2, .., 16 rows (64-element rows, 128-byte swizzle).
bool token_maps_m(CUtensorMap (&m)[kMMaxBoxes], const void* ptr, uint64_t inner, uint64_t rows,
                  int tn, bool f16) {
  bool ok = true;
  for (int b = 0; b < kMMaxBoxes; ++b)
    if ((tn >> b) >= 16) ok &= make_map(&m[b], ptr, inner, rows, (uint32_t)(tn >> b), f16);
  return ok;
}

// Row-major E4M3 matrix [rows, inner] read in boxes of 128 bytes x 128 rows
// with the 128-byte swizzle; rows past the end read as zero.
bool make_map_e4m3_sw128(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {128u, 128u};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool fp8_tm_supported(const moe_config_t& c) {
  const bool shared_ok = c.d_ff_shared == 0 || c.d_ff_shared % 128 == 0;
  return c.d_model % 256 == 0 && c.d_ff % 128 == 0 && shared_ok;
}

cudaError_t launch_rows_to_f16(const void* in, void* out, float* scale, int rows, int cols,
                               cudaStream_t s, LaunchCounter* lc) {
  if (rows == 0) return cudaSuccess;
  int blocks = (rows + 7) / 8;
  if (blocks > num_sms() * 8) blocks = num_sms() * 8;
  rows_to_f16_kernel<<<blocks, 256, 0, s>>>((const uint4*)in, (uint4*)out, scale, rows,
                                            cols / 8);
  count_launch(lc);
  return cudaGetLastError();
}

cudaError_t launch_gemm_fp8_tm(const moe_config_t& c, const ExpertArgs& a, int which, int tn,
                               cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  if (!fp8_tm_supported(c) || (tn != 32 && tn != 64 && tn != 128)) return cudaErrorInvalidValue;
  const bool f16 = a.tok_scale != nullptr;
  const int T = c.T, E = c.n_experts, d = c.d_model, F = c.d_ff, Fs = c.d_ff_shared;
  const int A = a.rows > 0 ? a.rows : T * c.top_k;
  const bool has_shared = Fs > 0 && a.ws_gate != nullptr;
  const moe_weight_scales_t& sc = *a.scales;
  MParams p{};
  bool ok = true;
  p.offsets = a.offsets;
  p.E = E;
  p.T = T;
  p.A = A;
  p.has_shared = has_shared ? 1 : 0;
  p.status = a.status;
  p.timeout_ns = kWaitTimeoutNs;
  p.perm = a.perm;
  p.perm_div = a.perm_div > 0 ? a.perm_div : 1;
  if (which == kGemmGateUp) {
    ok &= token_maps_m(p.a_map[0], a.x_perm, d, A, tn, f16);
    ok &= token_maps_m(p.a_map[1], a.x, d, T, tn, f16);
    p.row_scale[0] = a.tok_scale;
    p.row_scale[1] = a.tok_scale;
    ok &= make_map_e4m3_sw128(&p.b_map[0], a.w_gate, d, (uint64_t)E * F);
    ok &= make_map_e4m3_sw128(&p.u_map[0], a.w_up, d, (uint64_t)E * F);
    p.b_scale[0] = sc.gate_scale;
    p.u_scale[0] = sc.up_scale;
    if (has_shared) {
      ok &= make_map_e4m3_sw128(&p.b_map[1], a.ws_gate, d, Fs);
      ok &= make_map_e4m3_sw128(&p.u_map[1], a.ws_up, d, Fs);
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
    ok &= token_maps_m(p.a_map[0], a.h, F, A, tn, f16);
    ok &= make_map_e4m3_sw128(&p.b_map[0], a.w_down, F, (uint64_t)E * d);
    p.b_scale[0] = sc.down_scale;
    p.row_scale[0] = a.h_scale;
    p.row_scale[1] = a.hs_scale;
    if (has_shared) {
      ok &= token_maps_m(p.a_map[1], a.h_shared, Fs, T, tn, f16);
      ok &= make_map_e4m3_sw128(&p.b_map[1], a.ws_down, Fs, d);
      p.b_scale[1] = sc.shared_down_scale;
    } else {
      for (int b = 0; b < kMMaxBoxes; ++b) p.a_map[1][b] = p.a_map[0][b];
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
  cudaError_t err;
  const bool up = which == kGemmGateUp;
  if (f16) {
    if (tn == 32)
      err = up ? launch_m<kMGateUp, 32, true>(p, s) : launch_m<kMDown, 32, true>(p, s);
    else if (tn == 64)
      err = up ? launch_m<kMGateUp, 64, true>(p, s) : launch_m<kMDown, 64, true>(p, s);
    else
      err = up ? launch_m<kMGateUp, 128, true>(p, s) : launch_m<kMDown, 128, true>(p, s);
  } else {
    if (tn == 32)
      err = up ? launch_m<kMGateUp, 32, false>(p, s) : launch_m<kMDown, 32, false>(p, s);
    else if (tn == 64)
      err = up ? launch_m<kMGateUp, 64, false>(p, s) : launch_m<kMDown, 64, false>(p, s);
    else
      err = up ? launch_m<kMGateUp, 128, false>(p, s) : launch_m<kMDown, 128, false>(p, s);
  }
  count_launch(a.launches);
  return err;
}

}  // namespace moe

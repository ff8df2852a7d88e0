// Internal declarations shared by the library's translation units.
// Not part of the public ABI (that is include/moe_b300.h).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/moe_b300.h"

namespace moe {

// Device status word codes (first error wins; read by moe_get_error).
enum DeviceStatus : int32_t {
  kDevOk = 0,
  kDevTimeout = 1,     // a bounded wait ran out
  kDevBadIndex = 2,    // an index outside its valid range
};

__device__ __forceinline__ void record_error(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 32;
constexpr int kTopkMaxBlocks = 4 * 148;   // partial sums of the mean probability
constexpr int kDispatchChunk = 4096;      // assignments per dispatch block
constexpr int kDispatchThreads = 1024;

// Workspace layout: byte offsets from the workspace base, every region
// 1024-byte aligned.  A single function computes it for the host side.
struct WsLayout {
  size_t status;      // int32 status word
  size_t logits;      // [T, E] fp32
  size_t mp_partial;  // [kTopkMaxBlocks, E] fp32
  size_t topk_idx;    // [T, k] int32 (used when the caller passes no output)
  size_t topk_w;      // [T, k] fp32
  size_t counts;      // [E] int32
  size_t drops;       // [E] int32
  size_t offsets;     // [E + 1] int32
  size_t mean_prob;   // [E] fp32
  size_t block_hist;  // [nb, E] int32
  size_t block_base;  // [nb, E] int32
  size_t perm;        // [A] int32
  size_t row_of;      // [A] int32
  size_t drop_mask;   // [A] uint8
  size_t x_perm;      // [A, d] act
  size_t h;           // [A, F] act
  size_t h_shared;    // [T, F_s] act
  size_t y_perm;      // [A, d] fp32
  size_t y_shared;    // [T, d] fp32
  size_t shared_w;    // [T] fp32, per-token shared-expert gate
  size_t ec_scores;   // [E, T] fp32 (expert choice)
  size_t ec_w;        // [E, C] fp32 (expert choice)
  size_t ec_rowmap;   // [T, E] int32 (expert choice)
  size_t x16;         // [T, d] fp16 (E4M3 weights with fp16 operands)
  size_t tok_scale;   // [T] fp32
  size_t h_scale;     // [A] fp32
  size_t hs_scale;    // [T] fp32
  size_t total;
  int nb;             // dispatch blocks
};

WsLayout ws_layout(const moe_config_t& c);

// The shape and option rules every entry point applies to a configuration
// (MOE_OK, MOE_ERR_INVALID_ARG or MOE_ERR_UNSUPPORTED).
moe_status_t validate_config(const moe_config_t* c);

// Tokens each expert takes under expert-choice routing (at most T).
inline int ec_capacity(const moe_config_t& c) {
  long long C = c.capacity >= 0 ? (long long)c.capacity
                                : ((long long)c.T * c.top_k + c.n_experts - 1) / c.n_experts;
  if (C > c.T) C = c.T;
  return (int)C;
}
// Rows of the grouped (expert-major) buffers x_perm, h, y_perm and perm.
inline size_t grouped_rows(const moe_config_t& c) {
  if (c.routing == MOE_ROUTE_EXPERT_CHOICE) return (size_t)c.n_experts * (size_t)ec_capacity(c);
  return (size_t)c.T * (size_t)c.top_k;
}
constexpr int kEcMaxTokens = 32768;   // expert choice keeps one score column in shared memory

inline size_t act_bytes(const moe_config_t& c) { return c.act_dtype == MOE_BF16 ? 2 : 4; }

// Counts the library's own kernel launches of one call (for the benchmark's
// launch accounting).
struct LaunchCounter {
  int n = 0;
};
inline void count_launch(LaunchCounter* lc, int k = 1) {
  if (lc) lc->n += k;
}

// ---- launchers (each returns cudaGetLastError() after enqueueing) ----

// fp32 router logits held as `splits` partial sums [splits][T][E] plus an
// optional per-expert bias: z[t,e] = sum_s partials[s][t][e] (in s order) + bias[e].
// Streaming multiprocessors of the current device (queried once).
inline int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      n = 148;
  }
  return n;
}

struct LogitsView {
  const float* partials;
  int splits;
  size_t split_stride;   // elements from one partial to the next
  const float* bias;     // nullable
};

// Tensor-core router: one 128-token tile per CTA, reduction over d split
// across CTAs when there are few token tiles (at most kRouterCtaTarget CTAs
// unless T alone needs more).
constexpr int kRouterCtaTarget = 160;
constexpr int kMaxRouterSplits = 16;
struct RouterPlan {
  int m_tiles, kb_total, kb_per, splits;
};
RouterPlan plan_router(const moe_config_t& c);
// Floats of scratch the router needs for its partial sums.
inline size_t router_scratch_floats(const moe_config_t& c) {
  const size_t rows = (size_t)c.T > (size_t)kRouterCtaTarget * 128 ? (size_t)c.T
                                                                     : (size_t)kRouterCtaTarget * 128;
  return rows * (size_t)c.n_experts;
}

// Router logits of x . W^T (+ bias) into `scratch`; describes them in *view.
cudaError_t launch_router(const moe_config_t& c, const void* x, const void* w_router,
                          const float* bias, float* scratch, LogitsView* view, int32_t* status,
                          cudaStream_t s, LaunchCounter* lc = nullptr);
cudaError_t launch_router_tc(const moe_config_t& c, const void* x, const void* w_router,
                             float* partial, int32_t* status, cudaStream_t s,
                             LaunchCounter* lc = nullptr);

// Gating + top-k from logits; writes the summed logits to logits_out when
// given; mp_partial receives per-block partial sums of the scores, then a
// finalize kernel writes mean_prob (may be null).
// score_bias (nullable) and cfg.n_group / topk_group switch the ranking to
// s + b with group-limited selection (include/moe_b300.h, selection rule).
cudaError_t launch_topk(const moe_config_t& c, const LogitsView& z, const float* score_bias,
                        float* logits_out, int32_t* idx, float* w, float* mp_partial,
                        float* mean_prob, cudaStream_t s, LaunchCounter* lc = nullptr);

// out[t] = sigmoid(x_t . w), the per-token weight of the shared expert.
cudaError_t launch_shared_gate(const moe_config_t& c, const void* x, const void* w, float* out,
                               cudaStream_t s, LaunchCounter* lc = nullptr);

// *loss = alpha * E * sum_e f_e P_e, f_e = load_e / sum load (load = counts + drops).
cudaError_t launch_balance_loss(const moe_config_t& c, const int32_t* counts,
                                const int32_t* drops, const float* mean_prob, float alpha,
                                float* loss, cudaStream_t s);

// b_e -= gamma * sign(E * load_e - sum load), load = counts (+ drops).
cudaError_t launch_score_bias_update(const moe_config_t& c, const int32_t* counts,
                                     const int32_t* drops, float gamma, float* bias,
                                     cudaStream_t s);

// Dispatch: histogram, scan, stable scatter.  row_of may be null.
cudaError_t launch_dispatch(const moe_config_t& c, const int32_t* idx, int32_t* block_hist,
                            int32_t* block_base, int32_t* counts, int32_t* drops,
                            int32_t* offsets, int32_t* perm, int32_t* row_of,
                            uint8_t* drop_mask, int32_t* status, cudaStream_t s,
                            LaunchCounter* lc = nullptr);

// x_perm[r] = x[perm[r] / div] for r < offsets[E] (div = top_k: perm holds
// assignment ids; 1: perm holds tokens).
cudaError_t launch_gather(const moe_config_t& c, const void* x, const int32_t* perm,
                          const int32_t* offsets, void* x_perm, int32_t* status,
                          cudaStream_t s, LaunchCounter* lc = nullptr, int div = 0);

// Expert choice: scores, per-expert top-C selection (tokens / weights [E, C],
// offsets e*C, counts C, drops 0) and the mean probability.
// rowmap [T, E] (nullable): row of (t, e) in the grouped buffers, -1 if e did not take t.
cudaError_t launch_ec_route(const moe_config_t& c, const LogitsView& z, float* scores_t,
                            float* mp_partial, float* mean_prob, int32_t* tokens, float* weights,
                            int32_t* rowmap, int32_t* offsets, int32_t* counts, int32_t* drops,
                            cudaStream_t s, LaunchCounter* lc = nullptr);
// y[t] = sum over experts e that took t (ascending e) of w * y_perm[row] (+ w_s[t] y_shared[t]).
cudaError_t launch_ec_combine(const moe_config_t& c, const float* y_perm, const int32_t* rowmap,
                              const float* weights, const float* y_shared, const float* shared_w,
                              void* y, int32_t* status, cudaStream_t s,
                              LaunchCounter* lc = nullptr);
// mean_prob[e] = sum of the per-block partials / T (fixed order).
cudaError_t launch_mean_prob_finalize(const float* mp_partial, int nblocks, int E, int T,
                                      float* mean_prob, cudaStream_t s, LaunchCounter* lc);

// row_of[perm[r]] = r for r < offsets[E] (row_of pre-filled with -1).
cudaError_t launch_invert_perm(const moe_config_t& c, const int32_t* perm,
                               const int32_t* offsets, int32_t* row_of, int32_t* status,
                               cudaStream_t s, LaunchCounter* lc = nullptr);

// y[t] = sum_j kept g[t,j] y_perm[row_of[t*k+j]] (+ w_s[t] * y_shared[t], w_s = 1 when
// shared_w is null).
cudaError_t launch_combine(const moe_config_t& c, const float* y_perm, const float* topk_w,
                           const int32_t* row_of, const uint8_t* drop_mask,
                           const float* y_shared, const float* shared_w, void* y,
                           int32_t* status, cudaStream_t s, LaunchCounter* lc = nullptr);

// Grouped expert GEMMs.  Routed groups take rows offsets[e]..offsets[e+1] of
// x_perm / h; the shared group (when ws_* given) takes all T rows of x / h_shared.
struct ExpertArgs {
  const void* x;        // [T, d]
  const void* x_perm;   // [A, d], built by the gather in run_experts
  const int32_t* offsets;
  const int32_t* perm = nullptr;   // grouped row -> assignment (token choice) or token
  int perm_div = 0;                // perm[r] / perm_div is the token of grouped row r
  // E4M3 weights with fp16 operands: x, x_perm, h and h_shared hold fp16
  // rows, each row's values times its power-of-two scale below
  const float* tok_scale = nullptr;   // [T] per token (x, and x_perm through perm)
  const float* h_scale = nullptr;     // [A] per grouped row of h
  const float* hs_scale = nullptr;    // [T] per row of h_shared
  const void* w_gate; const void* w_up; const void* w_down;
  const void* ws_gate; const void* ws_up; const void* ws_down;
  void* h;              // [A, F]
  void* h_shared;       // [T, F_s]
  float* y_perm;        // [A, d]
  float* y_shared;      // [T, d]
  int32_t* status;
  const moe_weight_scales_t* scales = nullptr;   // E4M3 weights only
  int rows = 0;                                  // grouped rows (0: T * top_k)
  cudaEvent_t ev_up = nullptr;     // recorded before the gate/up GEMM when set (fp32 path)
  cudaEvent_t ev_down = nullptr;   // recorded before the down GEMM when set (fp32 path)
  LaunchCounter* launches = nullptr;
};

cudaError_t launch_experts_simt(const moe_config_t& c, const ExpertArgs& a, cudaStream_t s);
// One of the two bf16 grouped GEMMs (kGemmGateUp: x -> h, kGemmDown: h -> y),
// in one of two tile layouts:
//   _tc: tokens in the MMA's M (128-row token tiles, 256 weight rows per tile);
//   _wm: expert weights in M and tokens in N, on CTA pairs (token tiles of any
//        multiple of 32 rows, so ragged experts pad little).
constexpr int kGemmGateUp = 0;
constexpr int kGemmDown = 1;
cudaError_t launch_gemm_tc(const moe_config_t& c, const ExpertArgs& a, int which, cudaStream_t s);
cudaError_t launch_gemm_wm(const moe_config_t& c, const ExpertArgs& a, int which, cudaStream_t s);
// Tokens in M with E4M3 expert weights widened to bf16 on chip (a.scales set).
cudaError_t launch_gemm_fp8w(const moe_config_t& c, const ExpertArgs& a, int which,
                             cudaStream_t s);
// E4M3 weights in M, widened into tensor memory, token tiles of tn = 64 or
// 128 rows; needs fp8_tm_supported(c): d_model % 256, d_ff % 128 and
// d_ff_shared % 128 == 0.
bool fp8_tm_supported(const moe_config_t& c);
// rows x cols bf16 -> fp16 * 2^s per row (out may alias in), scale[r] = 2^s
// (rows_to_f16_kernel, experts_fp8_tm.cu); cols a multiple of 8.
cudaError_t launch_rows_to_f16(const void* in, void* out, float* scale, int rows, int cols,
                               cudaStream_t s, LaunchCounter* lc = nullptr);
cudaError_t launch_gemm_fp8_tm(const moe_config_t& c, const ExpertArgs& a, int which, int tn,
                               cudaStream_t s);

}  // namespace moe

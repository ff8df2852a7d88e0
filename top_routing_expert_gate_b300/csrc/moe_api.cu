// C ABI entry points (include/moe_b300.h): argument validation, workspace
// layout and the stream-ordered launch sequence of the layer forward.
#include "internal.cuh"

#include <math.h>
#include <stdlib.h>
#include <string.h>

namespace moe {

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

WsLayout ws_layout(const moe_config_t& c) {
  WsLayout L{};
  const size_t T = (size_t)c.T, E = (size_t)c.n_experts, k = (size_t)c.top_k;
  const size_t d = (size_t)c.d_model, F = (size_t)c.d_ff, Fs = (size_t)c.d_ff_shared;
  const size_t A = T * k;
  const size_t R = grouped_rows(c);   // rows of the expert-major buffers
  const bool ec = c.routing == MOE_ROUTE_EXPERT_CHOICE;
  const size_t ab = act_bytes(c);
  L.nb = (int)((A + kDispatchChunk - 1) / kDispatchChunk);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + (bytes ? bytes : 1), 1024);
    return at;
  };
  L.status = take(256);
  L.logits = take(router_scratch_floats(c) * 4);
  L.mp_partial = take((size_t)kTopkMaxBlocks * E * 4);
  L.topk_idx = take(A * 4);
  L.topk_w = take(A * 4);
  L.counts = take(E * 4);
  L.drops = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.mean_prob = take(E * 4);
  L.block_hist = take((size_t)L.nb * E * 4);
  L.block_base = take((size_t)L.nb * E * 4);
  L.perm = take(R * 4);
  L.row_of = take(A * 4);
  L.drop_mask = take(A);
  L.x_perm = take(R * d * ab);
  L.h = take(R * F * ab);
  L.h_shared = take(T * Fs * ab);
  L.y_perm = take(R * d * 4);
  L.y_shared = take(T * d * 4);
  L.shared_w = take(T * 4);
  L.ec_scores = take(ec ? E * T * 4 : 0);
  L.ec_w = take(ec ? R * 4 : 0);
  L.ec_rowmap = take(ec ? T * E * 4 : 0);
  const bool f8 = c.weight_format == MOE_WEIGHTS_FP8_E4M3;
  L.x16 = take(f8 ? T * d * 2 : 0);
  L.tok_scale = take(f8 ? T * 4 : 0);
  L.h_scale = take(f8 ? R * 4 : 0);
  L.hs_scale = take(f8 ? T * 4 : 0);
  L.total = o;
  return L;
}

}  // namespace moe

using namespace moe;

namespace {

template <typename P>
inline P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<char*>(ws) + off);
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Scratch the E4M3 weights-in-M kernel uses for fp16 operands (workspace).
struct F16Rows {
  void* x16 = nullptr;         // [T, d]
  float* tok_scale = nullptr;  // [T]
  float* h_scale = nullptr;    // [A]
  float* hs_scale = nullptr;   // [T]
};

F16Rows f16_rows(const moe_config_t& c, void* ws, const WsLayout& L) {
  F16Rows f;
  if (c.weight_format == MOE_WEIGHTS_FP8_E4M3) {
    f.x16 = at<char>(ws, L.x16);
    f.tok_scale = at<float>(ws, L.tok_scale);
    f.h_scale = at<float>(ws, L.h_scale);
    f.hs_scale = at<float>(ws, L.hs_scale);
  }
  return f;
}

// Shape/option checks shared by every call.
moe_status_t check_config(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->d_model <= 0 || c->n_experts < 1 || c->top_k < 1 ||
      c->top_k > c->n_experts || c->d_ff <= 0 || c->d_ff_shared < 0)
    return MOE_ERR_INVALID_ARG;
  if (c->gate != MOE_GATE_SOFTMAX && c->gate != MOE_GATE_SIGMOID) return MOE_ERR_INVALID_ARG;
  if ((c->act_dtype != MOE_BF16 && c->act_dtype != MOE_FP32) ||
      (c->out_dtype != MOE_BF16 && c->out_dtype != MOE_FP32))
    return MOE_ERR_INVALID_ARG;
  if (c->renormalize != 0 && c->renormalize != 1) return MOE_ERR_INVALID_ARG;
  if (!isfinite(c->routed_scaling_factor)) return MOE_ERR_INVALID_ARG;
  if ((long long)c->T * c->top_k > 0x7fffffffLL / 2) return MOE_ERR_INVALID_ARG;
  if (c->n_experts > kMaxExperts || c->top_k > kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if (c->d_model % 4 != 0) return MOE_ERR_UNSUPPORTED;
  if (c->act_dtype == MOE_BF16) {
    if (c->d_model % 64 != 0 || c->d_ff % 128 != 0 || c->d_ff_shared % 128 != 0)
      return MOE_ERR_UNSUPPORTED;
  }
  if (c->weight_format != MOE_WEIGHTS_ACT && c->weight_format != MOE_WEIGHTS_FP8_E4M3)
    return MOE_ERR_INVALID_ARG;
  if (c->routing != MOE_ROUTE_TOKEN_CHOICE && c->routing != MOE_ROUTE_EXPERT_CHOICE)
    return MOE_ERR_INVALID_ARG;
  if (c->routing == MOE_ROUTE_EXPERT_CHOICE) {
    if (c->n_group > 1) return MOE_ERR_INVALID_ARG;
    if (c->T > kEcMaxTokens) return MOE_ERR_UNSUPPORTED;
    if ((long long)c->n_experts * ec_capacity(*c) > 0x3fffffffLL) return MOE_ERR_INVALID_ARG;
  }
  if (c->weight_format == MOE_WEIGHTS_FP8_E4M3 && c->act_dtype != MOE_BF16)
    return MOE_ERR_UNSUPPORTED;
  // expert groups: 0 or 1 = none; otherwise equal groups of at least two
  // experts, at most 32 groups (one warp lane scores each group)
  if (c->n_group < 0) return MOE_ERR_INVALID_ARG;
  if (c->n_group > 1) {
    if (c->n_experts % c->n_group != 0 || c->n_experts / c->n_group < 2)
      return MOE_ERR_INVALID_ARG;
    if (c->n_group > 32) return MOE_ERR_UNSUPPORTED;
    if (c->topk_group < 1 || c->topk_group > c->n_group) return MOE_ERR_INVALID_ARG;
    if ((long long)c->top_k > (long long)c->topk_group * (c->n_experts / c->n_group))
      return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

moe_status_t check_ws(const moe_config_t* c, const void* ws, size_t ws_bytes) {
  if (!ws) return MOE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_WORKSPACE;
  if (ws_bytes < ws_layout(*c).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

// Required device pointer: non-null and 16-byte aligned (only when T > 0).
bool bad_ptr(const moe_config_t* c, const void* p) {
  if (c->T == 0) return false;
  return p == nullptr || !aligned16(p);
}
// Optional device pointer: null or 16-byte aligned.
bool bad_opt(const void* p) { return p != nullptr && !aligned16(p); }

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY_CUDA(expr)                         \
  do {                                             \
    cudaError_t _e = (expr);                       \
    if (_e != cudaSuccess) return MOE_ERR_CUDA;    \
  } while (0)

#define MOE_TRY(expr)                              \
  do {                                             \
    moe_status_t _s = (expr);                      \
    if (_s != MOE_OK) return _s;                   \
  } while (0)

// Tile layout of each bf16 grouped GEMM: true = expert weights in the MMA's
// M (launch_gemm_wm), false = tokens in M (launch_gemm_tc).
// MOE_B300_EXPERT_LAYOUT=tokens_m|weights_m|mixed overrides the choice for
// tests and tuning (mixed: weights in M for gate/up, tokens in M for down).
bool weights_in_m(const moe_config_t& c, int which) {
  (void)c;
  const char* o = getenv("MOE_B300_EXPERT_LAYOUT");
  if (o && strcmp(o, "tokens_m") == 0) return false;
  if (o && strcmp(o, "weights_m") == 0) return true;
  if (o && strcmp(o, "mixed") == 0) return which == kGemmGateUp;
  return false;
}

// E4M3 GEMM layout: the token-tile width of the weights-in-M kernel that
// widens into tensor memory (launch_gemm_fp8_tm: 32 or 64 for batches of a
// few tokens per expert, 128 for larger ones), or 0 for tokens in M
// (launch_gemm_fp8w).  The default takes 32 when the average expert gets at
// most 8 rows and the shared expert at most 64 (decode: every weight tile
// is streamed once, and the deeper widened-A ring keeps the MMAs off the
// critical path), 64 when the average expert gets at most 64 rows and the
// shared expert at most 256, else 128;
// MOE_B300_FP8_LAYOUT=tokens_m|weights_tm32|weights_tm|weights_tm128
// overrides it for tests and tuning.
int fp8_tmem_tile(const moe_config_t& c) {
  if (!fp8_tm_supported(c)) return 0;
  const char* o = getenv("MOE_B300_FP8_LAYOUT");
  if (o && strcmp(o, "tokens_m") == 0) return 0;
  if (o && strcmp(o, "weights_tm32") == 0) return 32;
  if (o && strcmp(o, "weights_tm") == 0) return 64;
  if (o && strcmp(o, "weights_tm128") == 0) return 128;
  const int64_t A = (int64_t)c.T * c.top_k;
  if (A <= (int64_t)8 * c.n_experts && c.T <= 64) return 32;
  return A <= (int64_t)64 * c.n_experts && c.T <= 256 ? 64 : 128;
}

// The gather (x_perm[r] = x[perm[r] / div]) and the two grouped GEMMs.  With
// E4M3 weights in the weights-in-M kernel the tokens become fp16 rows first
// (x, then h after gate/up), unless MOE_B300_FP8_TOKENS=bf16 (a test and
// tuning override) keeps the bf16 operands.
cudaError_t run_experts(const moe_config_t& c, ExpertArgs a, void* x_perm, cudaStream_t s,
                        const F16Rows& f16) {
  const bool fp8 = c.weight_format == MOE_WEIGHTS_FP8_E4M3;
  const int fp8_tn = fp8 ? fp8_tmem_tile(c) : 0;
  const int div = c.routing == MOE_ROUTE_EXPERT_CHOICE ? 1 : c.top_k;
  const char* tok_env = getenv("MOE_B300_FP8_TOKENS");
  const bool half_ops =
      fp8_tn > 0 && f16.x16 != nullptr && !(tok_env && strcmp(tok_env, "bf16") == 0);
  a.perm_div = div;
  if (half_ops) {
    const cudaError_t e =
        launch_rows_to_f16(a.x, f16.x16, f16.tok_scale, c.T, c.d_model, s, a.launches);
    if (e != cudaSuccess) return e;
    a.x = f16.x16;
    a.tok_scale = f16.tok_scale;
  }
  {
    const cudaError_t e = launch_gather(c, a.x, a.perm, a.offsets, x_perm, a.status, s,
                                        a.launches, div);
    if (e != cudaSuccess) return e;
    a.x_perm = x_perm;
  }
  if (c.act_dtype != MOE_BF16) return launch_experts_simt(c, a, s);
  for (int which = kGemmGateUp; which <= kGemmDown; ++which) {
    if (half_ops && which == kGemmDown) {
      // h and h_shared rewritten in place as fp16 rows
      cudaError_t e = launch_rows_to_f16(a.h, a.h, f16.h_scale, a.rows, c.d_ff, s, a.launches);
      if (e == cudaSuccess && a.ws_gate)
        e = launch_rows_to_f16(a.h_shared, a.h_shared, f16.hs_scale, c.T, c.d_ff_shared, s,
                               a.launches);
      if (e != cudaSuccess) return e;
      a.h_scale = f16.h_scale;
      a.hs_scale = f16.hs_scale;
    }
    cudaEvent_t ev = which == kGemmGateUp ? a.ev_up : a.ev_down;
    if (ev) {
      const cudaError_t e = cudaEventRecord(ev, s);
      if (e != cudaSuccess) return e;
    }
    const cudaError_t e = fp8_tn > 0              ? launch_gemm_fp8_tm(c, a, which, fp8_tn, s)
                          : fp8                   ? launch_gemm_fp8w(c, a, which, s)
                          : weights_in_m(c, which) ? launch_gemm_wm(c, a, which, s)
                                                   : launch_gemm_tc(c, a, which, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// E4M3 weights need every scale array of the weights in use; other formats none.
moe_status_t check_scales(const moe_config_t* c, const moe_weight_scales_t* sc,
                          bool has_shared) {
  if (c->weight_format != MOE_WEIGHTS_FP8_E4M3) return sc ? MOE_ERR_INVALID_ARG : MOE_OK;
  if (!sc) return MOE_ERR_INVALID_ARG;
  auto bad = [](const float* p) { return p == nullptr || !aligned16(p); };
  if (bad(sc->gate_scale) || bad(sc->up_scale) || bad(sc->down_scale)) return MOE_ERR_INVALID_ARG;
  if (has_shared && (bad(sc->shared_gate_scale) || bad(sc->shared_up_scale) ||
                     bad(sc->shared_down_scale)))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status_t check_shared_args(const moe_config_t* c, const void* g, const void* u,
                               const void* d) {
  const bool any = g || u || d;
  const bool all = g && u && d;
  if (any && !all) return MOE_ERR_INVALID_ARG;
  if (all && c->d_ff_shared == 0) return MOE_ERR_INVALID_ARG;
  if (!all && c->d_ff_shared > 0) return MOE_ERR_INVALID_ARG;
  if (bad_opt(g) || bad_opt(u) || bad_opt(d)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

}  // namespace

moe_status_t moe::validate_config(const moe_config_t* c) { return check_config(c); }

extern "C" {

int32_t moe_version(void) { return 500; }

const char* moe_status_string(moe_status_t st) {
  switch (st) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE";
  }
  return "MOE_ERR_UNKNOWN";
}

int32_t moe_capacity(int32_t T, int32_t E, double capacity_factor) {
  if (T < 0 || E <= 0 || !(capacity_factor >= 0.0)) return -1;
  const double c = ceil(((double)T / (double)E) * capacity_factor);
  if (c > 2147483647.0) return -1;
  return (int32_t)c;
}

int32_t moe_expert_choice_capacity(const moe_config_t* cfg) {
  if (check_config(cfg) != MOE_OK) return -1;
  return ec_capacity(*cfg);
}

moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* bytes) {
  MOE_TRY(check_config(cfg));
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = ws_layout(*cfg).total;
  return MOE_OK;
}

moe_status_t moe_workspace_init(const moe_config_t* cfg, void* ws, size_t ws_bytes,
                                void* stream) {
  MOE_TRY(check_config(cfg));
  MOE_TRY(check_ws(cfg, ws, ws_bytes));
  const WsLayout L = ws_layout(*cfg);
  return cuda_status(cudaMemsetAsync(at<char>(ws, L.status), 0, 256, (cudaStream_t)stream));
}

moe_status_t moe_topk_from_logits(const moe_config_t* cfg, const float* logits,
                                  const float* score_bias, int32_t* topk_idx, float* topk_w,
                                  float* mean_prob, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_config(cfg));
  if (cfg->routing != MOE_ROUTE_TOKEN_CHOICE) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(cfg, ws, ws_bytes));
  if (bad_ptr(cfg, logits) || bad_ptr(cfg, topk_idx) || bad_ptr(cfg, topk_w) ||
      bad_opt(mean_prob) || bad_opt(score_bias))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*cfg);
  const LogitsView view{logits, 1, 0, nullptr};
  return cuda_status(launch_topk(*cfg, view, score_bias, nullptr, topk_idx, topk_w,
                                 at<float>(ws, L.mp_partial), mean_prob, (cudaStream_t)stream));
}

moe_status_t moe_expert_choice_from_logits(const moe_config_t* cfg, const float* logits,
                                           int32_t* tokens, float* weights, float* mean_prob,
                                           void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_config(cfg));
  MOE_TRY(check_ws(cfg, ws, ws_bytes));
  if (cfg->routing != MOE_ROUTE_EXPERT_CHOICE) return MOE_ERR_INVALID_ARG;
  if (bad_ptr(cfg, logits) || bad_opt(mean_prob) ||
      (ec_capacity(*cfg) > 0 && (bad_ptr(cfg, tokens) || bad_ptr(cfg, weights))))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*cfg);
  const LogitsView view{logits, 1, 0, nullptr};
  return cuda_status(launch_ec_route(*cfg, view, at<float>(ws, L.ec_scores),
                                     at<float>(ws, L.mp_partial), mean_prob, tokens, weights,
                                     nullptr, at<int32_t>(ws, L.offsets),
                                     at<int32_t>(ws, L.counts), at<int32_t>(ws, L.drops),
                                     (cudaStream_t)stream));
}

moe_status_t moe_update_score_bias(const moe_config_t* cfg, const int32_t* counts,
                                   const int32_t* drops, float gamma, float* score_bias,
                                   void* stream) {
  MOE_TRY(check_config(cfg));
  if (!counts || !score_bias || !aligned16(counts) || !aligned16(score_bias) || bad_opt(drops))
    return MOE_ERR_INVALID_ARG;
  if (!isfinite(gamma)) return MOE_ERR_INVALID_ARG;
  return cuda_status(
      launch_score_bias_update(*cfg, counts, drops, gamma, score_bias, (cudaStream_t)stream));
}

moe_status_t moe_router_topk(const moe_config_t* cfg, const void* x, const void* w_router,
                             const float* router_bias, const float* score_bias,
                             float* logits_out, int32_t* topk_idx, float* topk_w,
                             float* mean_prob, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_config(cfg));
  if (cfg->routing != MOE_ROUTE_TOKEN_CHOICE) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(cfg, ws, ws_bytes));
  if (bad_ptr(cfg, x) || bad_ptr(cfg, w_router) || bad_ptr(cfg, topk_idx) ||
      bad_ptr(cfg, topk_w) || bad_opt(router_bias) || bad_opt(score_bias) ||
      bad_opt(logits_out) || bad_opt(mean_prob))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*cfg);
  cudaStream_t s = (cudaStream_t)stream;
  int32_t* status = at<int32_t>(ws, L.status);
  LogitsView view{};
  MOE_TRY_CUDA(launch_router(*cfg, x, w_router, router_bias, at<float>(ws, L.logits), &view,
                             status, s));
  return cuda_status(launch_topk(*cfg, view, score_bias, logits_out, topk_idx, topk_w,
                                 at<float>(ws, L.mp_partial), mean_prob, s));
}

moe_status_t moe_dispatch(const moe_config_t* cfg, const int32_t* topk_idx, int32_t* counts,
                          int32_t* drops, int32_t* offsets, int32_t* perm, uint8_t* drop_mask,
                          void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_config(cfg));
  if (cfg->routing != MOE_ROUTE_TOKEN_CHOICE) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(cfg, ws, ws_bytes));
  if (bad_ptr(cfg, topk_idx) || bad_ptr(cfg, perm) || bad_ptr(cfg, drop_mask) || !counts ||
      !drops || !offsets || !aligned16(counts) || !aligned16(drops) || !aligned16(offsets))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*cfg);
  return cuda_status(launch_dispatch(*cfg, topk_idx, at<int32_t>(ws, L.block_hist),
                                     at<int32_t>(ws, L.block_base), counts, drops, offsets,
                                     perm, nullptr, drop_mask, at<int32_t>(ws, L.status),
                                     (cudaStream_t)stream));
}

moe_status_t moe_grouped_swiglu(const moe_config_t* cfg, const void* x, const int32_t* perm,
                                const int32_t* offsets, const void* w_gate, const void* w_up,
                                const void* w_down, const void* ws_gate, const void* ws_up,
                                const void* ws_down, const moe_weight_scales_t* scales,
                                float* y_perm, float* y_shared, void* ws, size_t ws_bytes,
                                void* stream) {
  MOE_TRY(check_config(cfg));
  MOE_TRY(check_ws(cfg, ws, ws_bytes));
  if (bad_ptr(cfg, x) || bad_ptr(cfg, perm) || bad_ptr(cfg, w_gate) || bad_ptr(cfg, w_up) ||
      bad_ptr(cfg, w_down) || bad_ptr(cfg, y_perm) || !offsets || !aligned16(offsets))
    return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_shared_args(cfg, ws_gate, ws_up, ws_down));
  if ((ws_gate != nullptr) != (y_shared != nullptr) || bad_opt(y_shared))
    return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_scales(cfg, scales, ws_gate != nullptr));
  if (cfg->T == 0) return MOE_OK;
  const WsLayout L = ws_layout(*cfg);
  cudaStream_t s = (cudaStream_t)stream;
  int32_t* status = at<int32_t>(ws, L.status);
  ExpertArgs a{};
  a.x = x;
  a.offsets = offsets;
  a.perm = perm;
  a.w_gate = w_gate;
  a.w_up = w_up;
  a.w_down = w_down;
  a.ws_gate = ws_gate;
  a.ws_up = ws_up;
  a.ws_down = ws_down;
  a.h = at<char>(ws, L.h);
  a.h_shared = at<char>(ws, L.h_shared);
  a.y_perm = y_perm;
  a.y_shared = y_shared;
  a.status = status;
  a.scales = scales;
  a.rows = (int)grouped_rows(*cfg);
  return cuda_status(run_experts(*cfg, a, at<char>(ws, L.x_perm), s, f16_rows(*cfg, ws, L)));
}

moe_status_t moe_combine(const moe_config_t* cfg, const float* y_perm, const float* topk_w,
                         const int32_t* offsets, const int32_t* perm,
                         const uint8_t* drop_mask, const float* y_shared,
                         const float* shared_weight, void* y, void* ws, size_t ws_bytes,
                         void* stream) {
  MOE_TRY(check_config(cfg));
  if (cfg->routing != MOE_ROUTE_TOKEN_CHOICE) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(cfg, ws, ws_bytes));
  if (bad_ptr(cfg, y_perm) || bad_ptr(cfg, topk_w) || bad_ptr(cfg, perm) ||
      bad_ptr(cfg, drop_mask) || bad_ptr(cfg, y) || !offsets || !aligned16(offsets) ||
      bad_opt(y_shared) || bad_opt(shared_weight) || (shared_weight && !y_shared))
    return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  const WsLayout L = ws_layout(*cfg);
  cudaStream_t s = (cudaStream_t)stream;
  int32_t* status = at<int32_t>(ws, L.status);
  int32_t* row_of = at<int32_t>(ws, L.row_of);
  MOE_TRY_CUDA(launch_invert_perm(*cfg, perm, offsets, row_of, status, s));
  return cuda_status(launch_combine(*cfg, y_perm, topk_w, row_of, drop_mask, y_shared,
                                    shared_weight, y, status, s));
}

moe_status_t moe_shared_gate_weights(const moe_config_t* cfg, const void* x,
                                     const void* shared_gate, float* weights, void* stream) {
  MOE_TRY(check_config(cfg));
  if (bad_ptr(cfg, x) || bad_ptr(cfg, weights) || !shared_gate || !aligned16(shared_gate))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_shared_gate(*cfg, x, shared_gate, weights, (cudaStream_t)stream));
}

moe_status_t moe_balance_loss(const moe_config_t* cfg, const int32_t* counts,
                              const int32_t* drops, const float* mean_prob, float alpha,
                              float* loss, void* stream) {
  MOE_TRY(check_config(cfg));
  if (!counts || !mean_prob || !loss || !aligned16(counts) || !aligned16(mean_prob) ||
      bad_opt(drops) || ((uintptr_t)loss & 3u) != 0 || !isfinite(alpha))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(
      launch_balance_loss(*cfg, counts, drops, mean_prob, alpha, loss, (cudaStream_t)stream));
}

}  // extern "C"

namespace {

// The layer forward.  When `ev` is non-null, ev[i] is recorded on the stream
// before stage i (MOE_NUM_STAGES stages) and ev[MOE_NUM_STAGES] after the last.
moe_status_t layer_forward_impl(const moe_config_t* cfg, const void* x, const void* w_router,
                                const float* router_bias, const float* score_bias,
                                const void* w_gate, const void* w_up,
                                const void* w_down, const void* ws_gate, const void* ws_up,
                                const void* ws_down, const void* shared_gate,
                                const moe_weight_scales_t* scales, void* y,
                                int32_t* topk_idx, float* topk_w, int32_t* counts,
                                int32_t* drops, float* mean_prob, void* ws, size_t ws_bytes,
                                void* stream, cudaEvent_t* ev, int32_t* n_launches) {
  MOE_TRY(check_config(cfg));
  MOE_TRY(check_ws(cfg, ws, ws_bytes));
  if (bad_ptr(cfg, x) || bad_ptr(cfg, w_router) || bad_ptr(cfg, w_gate) ||
      bad_ptr(cfg, w_up) || bad_ptr(cfg, w_down) || bad_ptr(cfg, y) || bad_opt(router_bias) ||
      bad_opt(score_bias) ||
      bad_opt(topk_idx) || bad_opt(topk_w) || bad_opt(counts) || bad_opt(drops) ||
      bad_opt(mean_prob))
    return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_shared_args(cfg, ws_gate, ws_up, ws_down));
  if (bad_opt(shared_gate) || (shared_gate && !ws_gate)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_scales(cfg, scales, ws_gate != nullptr));
  const bool ec = cfg->routing == MOE_ROUTE_EXPERT_CHOICE;
  if (ec && (topk_idx || topk_w || score_bias)) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*cfg);
  cudaStream_t s = (cudaStream_t)stream;
  const moe_config_t& c = *cfg;
  LaunchCounter lc;
  auto mark = [&](int i) -> cudaError_t {
    return ev ? cudaEventRecord(ev[i], s) : cudaSuccess;
  };
  if (c.T == 0) {
    if (counts) MOE_TRY_CUDA(cudaMemsetAsync(counts, 0, 4 * (size_t)c.n_experts, s));
    if (drops) MOE_TRY_CUDA(cudaMemsetAsync(drops, 0, 4 * (size_t)c.n_experts, s));
    if (mean_prob) MOE_TRY_CUDA(cudaMemsetAsync(mean_prob, 0, 4 * (size_t)c.n_experts, s));
    for (int i = 0; ev && i <= MOE_NUM_STAGES; ++i) MOE_TRY_CUDA(mark(i));
    if (n_launches) *n_launches = 0;
    return MOE_OK;
  }
  int32_t* status = at<int32_t>(ws, L.status);
  int32_t* idx = topk_idx ? topk_idx : at<int32_t>(ws, L.topk_idx);
  float* g = topk_w ? topk_w : at<float>(ws, L.topk_w);
  int32_t* cnt = counts ? counts : at<int32_t>(ws, L.counts);
  int32_t* drp = drops ? drops : at<int32_t>(ws, L.drops);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* perm = at<int32_t>(ws, L.perm);
  int32_t* row_of = at<int32_t>(ws, L.row_of);
  uint8_t* dmask = at<uint8_t>(ws, L.drop_mask);
  float* z = at<float>(ws, L.logits);

  MOE_TRY_CUDA(mark(MOE_STAGE_ROUTER));
  LogitsView view{};
  MOE_TRY_CUDA(launch_router(c, x, w_router, router_bias, z, &view, status, s, &lc));
  float* shared_w = shared_gate ? at<float>(ws, L.shared_w) : nullptr;
  if (shared_gate) MOE_TRY_CUDA(launch_shared_gate(c, x, shared_gate, shared_w, s, &lc));
  MOE_TRY_CUDA(mark(MOE_STAGE_TOPK));
  float* ec_w = at<float>(ws, L.ec_w);
  if (ec) {
    // expert choice: scores and the per-expert selection give perm (tokens,
    // expert-major, ascending), the weights and offsets e*C directly
    MOE_TRY_CUDA(launch_ec_route(c, view, at<float>(ws, L.ec_scores), at<float>(ws, L.mp_partial),
                                 mean_prob, perm, ec_w, at<int32_t>(ws, L.ec_rowmap), offsets, cnt,
                                 drp, s, &lc));
    MOE_TRY_CUDA(mark(MOE_STAGE_DISPATCH));
  } else {
    MOE_TRY_CUDA(launch_topk(c, view, score_bias, nullptr, idx, g, at<float>(ws, L.mp_partial),
                             mean_prob, s, &lc));
    MOE_TRY_CUDA(mark(MOE_STAGE_DISPATCH));
    MOE_TRY_CUDA(launch_dispatch(c, idx, at<int32_t>(ws, L.block_hist),
                                 at<int32_t>(ws, L.block_base), cnt, drp, offsets, perm, row_of,
                                 dmask, status, s, &lc));
  }
  MOE_TRY_CUDA(mark(MOE_STAGE_GATHER));
  const bool has_shared = ws_gate != nullptr;
  ExpertArgs a{};
  a.x = x;
  a.offsets = offsets;
  a.perm = perm;
  a.w_gate = w_gate;
  a.w_up = w_up;
  a.w_down = w_down;
  a.ws_gate = ws_gate;
  a.ws_up = ws_up;
  a.ws_down = ws_down;
  a.h = at<char>(ws, L.h);
  a.h_shared = at<char>(ws, L.h_shared);
  a.y_perm = at<float>(ws, L.y_perm);
  a.y_shared = has_shared ? at<float>(ws, L.y_shared) : nullptr;
  a.status = status;
  a.scales = scales;
  a.rows = (int)grouped_rows(c);
  a.ev_up = ev ? ev[MOE_STAGE_GATE_UP] : nullptr;
  a.ev_down = ev ? ev[MOE_STAGE_DOWN] : nullptr;
  a.launches = &lc;
  MOE_TRY_CUDA(run_experts(c, a, at<char>(ws, L.x_perm), s, f16_rows(c, ws, L)));
  MOE_TRY_CUDA(mark(MOE_STAGE_COMBINE));
  if (ec)
    MOE_TRY_CUDA(launch_ec_combine(c, a.y_perm, at<int32_t>(ws, L.ec_rowmap), ec_w, a.y_shared,
                                   shared_w, y, status, s, &lc));
  else
    MOE_TRY_CUDA(
        launch_combine(c, a.y_perm, g, row_of, dmask, a.y_shared, shared_w, y, status, s, &lc));
  MOE_TRY_CUDA(mark(MOE_NUM_STAGES));
  if (n_launches) *n_launches = lc.n;
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status_t moe_layer_forward(const moe_config_t* cfg, const void* x, const void* w_router,
                               const float* router_bias, const float* score_bias,
                               const void* w_gate, const void* w_up,
                               const void* w_down, const void* ws_gate, const void* ws_up,
                               const void* ws_down, const void* shared_gate,
                               const moe_weight_scales_t* scales, void* y,
                               int32_t* topk_idx, float* topk_w, int32_t* counts,
                               int32_t* drops, float* mean_prob, void* ws, size_t ws_bytes,
                               void* stream) {
  return layer_forward_impl(cfg, x, w_router, router_bias, score_bias, w_gate, w_up, w_down,
                            ws_gate, ws_up, ws_down, shared_gate, scales, y, topk_idx, topk_w,
                            counts, drops, mean_prob, ws, ws_bytes, stream, nullptr, nullptr);
}

moe_status_t moe_layer_forward_host(const moe_config_t* cfg, const void* x_host, void* x,
                                    const void* w_router, const float* router_bias,
                                    const float* score_bias, const void* w_gate,
                                    const void* w_up, const void* w_down, const void* ws_gate,
                                    const void* ws_up, const void* ws_down,
                                    const void* shared_gate, const moe_weight_scales_t* scales,
                                    void* y, void* y_host, int32_t* topk_idx, float* topk_w,
                                    int32_t* counts, int32_t* drops, float* mean_prob, void* ws,
                                    size_t ws_bytes, void* stream) {
  MOE_TRY(check_config(cfg));
  MOE_TRY(check_ws(cfg, ws, ws_bytes));
  if (cfg->T > 0 && (x_host == nullptr || y_host == nullptr || bad_ptr(cfg, x) || bad_ptr(cfg, y)))
    return MOE_ERR_INVALID_ARG;
  const cudaStream_t s = (cudaStream_t)stream;
  const size_t n = (size_t)cfg->T * cfg->d_model;
  if (n > 0)
    MOE_TRY_CUDA(cudaMemcpyAsync(x, x_host, n * act_bytes(*cfg), cudaMemcpyHostToDevice, s));
  MOE_TRY(layer_forward_impl(cfg, x, w_router, router_bias, score_bias, w_gate, w_up, w_down,
                             ws_gate, ws_up, ws_down, shared_gate, scales, y, topk_idx, topk_w,
                             counts, drops, mean_prob, ws, ws_bytes, stream, nullptr, nullptr));
  const size_t yb = cfg->out_dtype == MOE_BF16 ? 2 : 4;
  if (n > 0) MOE_TRY_CUDA(cudaMemcpyAsync(y_host, y, n * yb, cudaMemcpyDeviceToHost, s));
  return MOE_OK;
}

moe_status_t moe_layer_forward_profiled(const moe_config_t* cfg, const void* x,
                                        const void* w_router, const float* router_bias,
                                        const float* score_bias, const void* w_gate,
                                        const void* w_up, const void* w_down,
                                        const void* ws_gate, const void* ws_up,
                                        const void* ws_down, const void* shared_gate,
                                        const moe_weight_scales_t* scales, void* y,
                                        int32_t* topk_idx, float* topk_w, int32_t* counts,
                                        int32_t* drops, float* mean_prob, void* ws,
                                        size_t ws_bytes, void* stream, void** stage_events,
                                        int32_t* n_launches) {
  if (!stage_events) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i <= MOE_NUM_STAGES; ++i)
    if (!stage_events[i]) return MOE_ERR_INVALID_ARG;
  return layer_forward_impl(cfg, x, w_router, router_bias, score_bias, w_gate, w_up, w_down,
                            ws_gate, ws_up, ws_down, shared_gate, scales, y, topk_idx, topk_w,
                            counts, drops, mean_prob, ws, ws_bytes, stream,
                            (cudaEvent_t*)stage_events, n_launches);
}

moe_status_t moe_get_error(const void* ws, void* stream) {
  if (!ws) return MOE_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  int32_t host = 0;
  int32_t* dev = (int32_t*)ws;   // the status word is the first region (offset 0)
  if (cudaMemcpyAsync(&host, dev, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (host != 0) {
    if (cudaMemsetAsync(dev, 0, sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (host == kDevTimeout) return MOE_ERR_TIMEOUT;
  if (host != 0) return MOE_ERR_DEVICE;
  return MOE_OK;
}

}  // extern "C"

/*
 * moe_b300.h - C ABI of the single-GPU MoE FFN layer forward (NVIDIA B300,
 * sm_103a).
 *
 * The layer, as the pages state it:
 *   logits = x . W_router^T                     ("10. 混合专家 MoE：总参数与激活参数",
 *                                                 niuwancheng.cn, block sketch in
 *                                                 "把一个大 FFN 换成一组小 FFN")
 *   score  = softmax(logits) or sigmoid(logits) (same page, "路由器怎样选专家：
 *                                                 top-k 与两种门控")
 *   top-k on the logits; weights renormalised over the chosen k and times
 *   routed_scaling_factor (same section)
 *   capacity = ceil((T / E) * capacity_factor); over-capacity assignments are
 *   dropped and ride the residual (same page, "负载不均：路由坍缩与丢 token")
 *   y_t = sum_{i in TopK} g_{t,i} E_i(x_t) + S(x_t)   ("MoE为什么只激活一部分专家",
 *                                                 hi-bin.com, "Router 怎样给 Token
 *                                                 选专家"; shared expert S from
 *                                                 "细粒度专家与共享专家")
 *   E_i(x) = (SiLU(x W_gate,i^T) * (x W_up,i^T)) W_down,i^T
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *     never allocates device memory: each call takes a workspace `ws` of at
 *     least moe_workspace_size() bytes, 256-byte aligned, zero-filled once
 *     before its first use (moe_workspace_init does this).  One workspace must
 *     not be used by two calls that may run concurrently.
 *   - Every compute call is asynchronous on the caller's `stream` (a
 *     cudaStream_t passed as void*, NULL = the legacy default stream).  No call
 *     synchronises the stream or copies device data to the host, except
 *     moe_get_error.
 *   - Argument errors are detected on the host before anything is enqueued and
 *     returned synchronously; nothing is launched then.  Launch errors return
 *     MOE_ERR_CUDA.  Errors found by kernels (a bounded wait that ran out, an
 *     index out of range) are recorded in a status word inside `ws` and
 *     reported by moe_get_error.
 *   - Layouts are row-major with nn.Linear orientation (out x in):
 *       x [T, d], w_router [E, d], w_gate / w_up [E, F, d], w_down [E, d, F],
 *       ws_gate / ws_up [F_s, d], ws_down [d, F_s].
 *     Activations and weights have dtype act_dtype (MOE_BF16 or MOE_FP32);
 *     accumulation is always fp32.  Logits, weights and statistics are fp32.
 *   - Assignment a = t * top_k + j is token t's j-th choice (j = 0 best).
 *   - Pointers must be 16-byte aligned.  For MOE_BF16, d_model must be a
 *     multiple of 64 and d_ff / d_ff_shared multiples of 128 (the tensor-core
 *     tiles); otherwise MOE_ERR_UNSUPPORTED.  1 <= top_k <= n_experts <= 256.
 *   - No C++ exception crosses this boundary.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misalignment, k > E  */
  MOE_ERR_UNSUPPORTED = 2,  /* valid but outside what the kernels implement */
  MOE_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed            */
  MOE_ERR_WORKSPACE = 4,    /* workspace null or too small                  */
  MOE_ERR_TIMEOUT = 5,      /* a kernel's bounded wait ran out (moe_get_error) */
  MOE_ERR_DEVICE = 6        /* a kernel found an inconsistent index (moe_get_error) */
} moe_status_t;

typedef enum { MOE_GATE_SOFTMAX = 0, MOE_GATE_SIGMOID = 1 } moe_gate_t;
typedef enum { MOE_BF16 = 0, MOE_FP32 = 1 } moe_dtype_t;
/* Storage of the routed and shared expert weights (the router weight is
 * always act_dtype).  MOE_WEIGHTS_FP8_E4M3: each weight is an 8-bit E4M3 code
 * (1 sign, 4 exponent bits of bias 7, 3 mantissa bits; max 448; NaN codes out
 * of contract) times an fp32 scale of its output channel
 * (moe_weight_scales_t) - "10. 混合专家 MoE", section "推理时": DeepSeek-V3
 * ships FP8 weights, about one byte per parameter.  Requires act_dtype
 * MOE_BF16; the products are exact in bf16 and the scale is applied to the
 * fp32 accumulator of each output. */
typedef enum { MOE_WEIGHTS_ACT = 0, MOE_WEIGHTS_FP8_E4M3 = 1 } moe_weight_format_t;
/* Who chooses.  MOE_ROUTE_TOKEN_CHOICE: each token takes its top_k experts
 * (selection rule below).  MOE_ROUTE_EXPERT_CHOICE (the amazingdata.cn
 * article on MoE routing, paragraph on expert choice: each expert takes a
 * fixed number of the tokens it scores highest, which balances the load by
 * construction; a token may be taken by no expert): expert e takes the C = moe_expert_choice_capacity(cfg)
 * tokens with the largest fp32 score s[t, e] (ties to the lower token), and
 * y_t = sum over the experts that took t of s[t, e] * E_e(x_t) (+ shared). */
typedef enum { MOE_ROUTE_TOKEN_CHOICE = 0, MOE_ROUTE_EXPERT_CHOICE = 1 } moe_routing_t;

/* Layer description.  All fields are plain 32-bit values. */
typedef struct {
  int32_t T;              /* tokens in the batch, >= 0                          */
  int32_t d_model;        /* d                                                  */
  int32_t n_experts;      /* E, routed experts, 1..256                          */
  int32_t top_k;          /* k, 1..E                                            */
  int32_t d_ff;           /* F, routed expert SwiGLU width                      */
  int32_t d_ff_shared;    /* F_s, shared expert width; 0 = no shared expert     */
  int32_t gate;           /* moe_gate_t                                         */
  int32_t renormalize;    /* 1: g_j = score_j / sum_chosen score; 0: g_j = score_j */
  float routed_scaling_factor; /* multiplies every routed weight (1.0, or 2.5)  */
  int32_t capacity;       /* < 0: unlimited; >= 0: kept slots per expert (0 drops all) */
  int32_t act_dtype;      /* moe_dtype_t of x, weights and the expert activations */
  int32_t out_dtype;      /* moe_dtype_t of y                                   */
  int32_t n_group;        /* expert groups for group-limited selection; 0 or 1 = none.
                             Otherwise 2..32, dividing n_experts into groups of >= 2 */
  int32_t topk_group;     /* groups kept per token when n_group > 1 (1..n_group;
                             top_k <= topk_group * n_experts / n_group)           */
  int32_t weight_format;  /* moe_weight_format_t of the expert weights          */
  int32_t routing;        /* moe_routing_t; expert choice requires T <= 32768, no
                             score bias or groups, and no topk_idx / topk_w outputs */
} moe_config_t;

/* Per-output-channel scales of E4M3 expert weights (weight_format ==
 * MOE_WEIGHTS_FP8_E4M3): weight[row, c] = e4m3(code[row, c]) * scale[row].
 * Device fp32 arrays, 16-byte aligned.  Pass NULL for MOE_WEIGHTS_ACT. */
typedef struct {
  const float* gate_scale;         /* [E, F] (rows of w_gate)                */
  const float* up_scale;           /* [E, F] (rows of w_up)                  */
  const float* down_scale;         /* [E, d] (rows of w_down)                */
  const float* shared_gate_scale;  /* [F_s]; NULL without a shared expert    */
  const float* shared_up_scale;    /* [F_s]                                   */
  const float* shared_down_scale;  /* [d]                                     */
} moe_weight_scales_t;

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
MOE_API int32_t moe_version(void);

/* Human-readable name of a status code (static storage). */
MOE_API const char* moe_status_string(moe_status_t st);

/* Expert capacity ceil((T / E) * capacity_factor), computed in IEEE double in
 * that order ("负载不均：路由坍缩与丢 token": 2 x 1.25 = 2.5 is rounded up to 3).
 * Returns -1 for T < 0, E <= 0 or capacity_factor < 0 (or NaN). */
MOE_API int32_t moe_capacity(int32_t T, int32_t E, double capacity_factor);

/* Tokens each expert takes under expert-choice routing: cfg->capacity when
 * >= 0, else ceil(T * top_k / E) (as many slots as token choice fills on
 * average), at most T.  -1 for an invalid configuration. */
MOE_API int32_t moe_expert_choice_capacity(const moe_config_t* cfg);

/* Bytes of workspace every call below needs for this configuration. */
MOE_API moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* bytes);

/* Clears the workspace's device status word (cudaMemsetAsync on `stream`).
 * Call once after allocating the workspace. */
MOE_API moe_status_t moe_workspace_init(const moe_config_t* cfg, void* ws, size_t ws_bytes,
                                void* stream);

/* Selection rule shared by moe_router_topk, moe_topk_from_logits and the
 * layer forward.  Scores are s = softmax(z) or sigmoid(z) of the fp32 logits.
 *   - score_bias == NULL and n_group <= 1: the k largest LOGITS are chosen
 *     (the same experts as the k largest scores), ties to the lower index.
 *   - otherwise (DeepSeek-V3 auxiliary-loss-free routing, "10. 混合专家 MoE",
 *     section "DeepSeek-V3 的无辅助损失偏置"): the ranking key is
 *     s_e + score_bias[e] (fp32; bias 0 when NULL).  With n_group > 1 the
 *     experts form n_group consecutive groups of E / n_group, a group's score
 *     is the sum of its two largest keys, the topk_group best groups are kept
 *     (ties to the lower group) and the k largest keys among their experts
 *     are chosen (ties to the lower index).  The combine weights use the raw
 *     scores s, never the bias.
 * topk_idx lists the chosen experts by ranking key, descending. */

/* Router + gating + top-k (the block sketch's first four lines).
 *   x [T, d] act_dtype; w_router [E, d] act_dtype;
 *   router_bias [E] fp32 or NULL: added to every logit before scoring and
 *     selection (used by the Zipf-skewed Switch-style layer);
 *   score_bias [E] fp32 or NULL: selection-only bias on the scores (see the
 *     selection rule above; DeepSeek-V3's e_score_correction_bias);
 *   logits_out [T, E] fp32 or NULL: the logits incl. bias;
 *   topk_idx [T, k] int32: chosen experts, logit descending, ties to the
 *     lower expert index;
 *   topk_w [T, k] fp32: combine weights (renormalised and scaled per cfg);
 *   mean_prob [E] fp32 or NULL: (1/T) sum_t score[t, e] over ALL experts
 *     (softmax probability or sigmoid score), reduced in a fixed order. */
MOE_API moe_status_t moe_router_topk(const moe_config_t* cfg, const void* x, const void* w_router,
                             const float* router_bias, const float* score_bias,
                             float* logits_out,
                             int32_t* topk_idx, float* topk_w, float* mean_prob,
                             void* ws, size_t ws_bytes, void* stream);

/* Gating + top-k from caller-supplied fp32 logits [T, E] (router bias
 * already in), with the optional selection-only score_bias [E].  Outputs as
 * moe_router_topk.  Without score bias or groups the selection compares fp32
 * logits only, so it is reproducible bit for bit from the same logits; with
 * them it compares fp32 s + b, which depends on the fp32 exp. */
MOE_API moe_status_t moe_topk_from_logits(const moe_config_t* cfg, const float* logits,
                                  const float* score_bias,
                                  int32_t* topk_idx, float* topk_w, float* mean_prob,
                                  void* ws, size_t ws_bytes, void* stream);

/* Expert-choice selection from fp32 logits [T, E] (cfg->routing must be
 * MOE_ROUTE_EXPERT_CHOICE; C = moe_expert_choice_capacity(cfg)):
 *   tokens [E, C] int32: expert e's tokens in ascending order;
 *   weights [E, C] fp32: s[tokens[e, i], e], the combine weights;
 *   mean_prob [E] fp32 or NULL: (1/T) sum_t s[t, e].
 * The selection compares fp32 scores (softmax or sigmoid of the logits). */
MOE_API moe_status_t moe_expert_choice_from_logits(const moe_config_t* cfg, const float* logits,
                                                   int32_t* tokens, float* weights,
                                                   float* mean_prob, void* ws, size_t ws_bytes,
                                                   void* stream);

/* One step of the auxiliary-loss-free bias ("DeepSeek-V3 的无辅助损失偏置":
 * after each batch an overloaded expert's bias is lowered by gamma and an
 * underloaded one's raised by gamma):
 *   load[e] = counts[e] + drops[e]  (drops may be NULL),
 *   score_bias[e] -= gamma * sign(E * load[e] - sum_e' load[e'])
 * i.e. compared with the mean load exactly, in integers; an expert exactly
 * at the mean keeps its bias.  counts, drops: [E] int32 device (as written
 * by moe_dispatch or the layer forward); score_bias: [E] fp32 device,
 * updated in place.  One small kernel on `stream`. */
MOE_API moe_status_t moe_update_score_bias(const moe_config_t* cfg, const int32_t* counts,
                                           const int32_t* drops, float gamma, float* score_bias,
                                           void* stream);

/* Capacity + dispatch ("负载不均：路由坍缩与丢 token"; the block sketch's
 * per-expert grouping).  Assignments are visited in ascending a; each takes
 * the next free slot of its expert or is dropped once the expert holds
 * cfg->capacity.  Deterministic (no order-dependent atomics).
 *   topk_idx [T, k] int32 (values in [0, E); others -> MOE_ERR_DEVICE);
 *   counts [E] int32: kept assignments per expert;
 *   drops [E] int32: dropped assignments per expert;
 *   offsets [E + 1] int32: exclusive prefix sum of counts;
 *   perm [T * k] int32: perm[offsets[e] + slot] = a; entries at and beyond
 *     offsets[E] are left unspecified;
 *   drop_mask [T * k] uint8: 1 where assignment a was dropped. */
MOE_API moe_status_t moe_dispatch(const moe_config_t* cfg, const int32_t* topk_idx,
                          int32_t* counts, int32_t* drops, int32_t* offsets,
                          int32_t* perm, uint8_t* drop_mask,
                          void* ws, size_t ws_bytes, void* stream);

/* The same dispatch as moe_dispatch, for callers that cannot allocate device
 * memory: no workspace argument, and nothing is allocated by this call.  The
 * pages have no counterpart of this entry point; it exists for callers whose
 * device memory is planned and owned by someone else (a host framework or
 * runtime that fixes its memory arena when a model is loaded and rejects or
 * cannot satisfy allocations afterwards, or a latency-critical serving loop
 * where cudaMalloc/cudaFree would stall on the device), so neither they nor
 * this library may call cudaMalloc to obtain a workspace.
 *   - Scratch: the per-block tables live in a fixed 64 KiB device array built
 *     into the library, held on every GPU that loads it until the process
 *     exits.  Limit: T * top_k <= 131072 assignments (and n_experts <= 256);
 *     larger batches return MOE_ERR_UNSUPPORTED without launching anything.
 *   - Every call looks up that array's device address on the current
 *     device (cudaGetSymbolAddress, a host-side lookup), so the address stays
 *     right after cudaDeviceReset.  The first call on a device may also load
 *     the library's device code there; make that first call before any
 *     stream capture.
 *   - All calls in the process share the one array: calls whose GPU work may
 *     overlap (different streams, or different host threads on one device)
 *     race on it and must be serialised by the caller.
 *   - There is no status word: an expert index outside [0, E) is not counted
 *     anywhere and its assignment is marked dropped, so sum(counts) +
 *     sum(drops) < T * top_k reveals it.
 * Arguments, configuration rules (token-choice routing only), outputs and
 * determinism are those of moe_dispatch. */
MOE_API moe_status_t moe_dispatch_no_workspace(const moe_config_t* cfg, const int32_t* topk_idx,
                                               int32_t* counts, int32_t* drops,
                                               int32_t* offsets, int32_t* perm,
                                               uint8_t* drop_mask, void* stream);

/* Grouped SwiGLU experts over dispatched rows (the grouped GEMM that replaces
 * the block sketch's per-expert loop).  Row r < offsets[E] of the grouped
 * batch is token perm[r] / k and belongs to the expert whose segment holds r:
 *   y_perm[r, :] = E_e(x[perm[r] / k, :])            fp32 [T * k, d]
 * Rows at and beyond offsets[E] are left unspecified.  Expert weights are
 * act_dtype, or E4M3 codes with `scales` when cfg->weight_format is
 * MOE_WEIGHTS_FP8_E4M3 (scales must be NULL otherwise).  If the shared expert
 * weights are given (cfg->d_ff_shared > 0), also
 *   y_shared[t, :] = S(x[t, :])                      fp32 [T, d]
 * ws_gate/ws_up/ws_down/y_shared must all be NULL when d_ff_shared == 0. */
MOE_API moe_status_t moe_grouped_swiglu(const moe_config_t* cfg, const void* x,
                                const int32_t* perm, const int32_t* offsets,
                                const void* w_gate, const void* w_up, const void* w_down,
                                const void* ws_gate, const void* ws_up, const void* ws_down,
                                const moe_weight_scales_t* scales,
                                float* y_perm, float* y_shared,
                                void* ws, size_t ws_bytes, void* stream);

/* Weighted unpermute-combine:
 *   y[t, :] = sum_{j: drop_mask[t*k+j] == 0} topk_w[t, j] * y_perm[row(t*k+j), :]
 *             + w_s[t] * y_shared[t, :]   (if y_shared != NULL)
 * where row(a) is the r with perm[r] == a and w_s[t] = shared_weight[t]
 * (fp32 [T], e.g. from moe_shared_gate_weights) or 1 when shared_weight is
 * NULL (shared_weight requires y_shared).  Summed in fp32 in ascending j,
 * then the shared term; written once as out_dtype.  Tokens whose choices were
 * all dropped get the shared term or 0: y excludes the residual. */
MOE_API moe_status_t moe_combine(const moe_config_t* cfg, const float* y_perm, const float* topk_w,
                         const int32_t* offsets, const int32_t* perm,
                         const uint8_t* drop_mask, const float* y_shared,
                         const float* shared_weight, void* y,
                         void* ws, size_t ws_bytes, void* stream);

/* Per-token weight of the shared expert, weights[t] = sigmoid(x_t . w)
 * ("10. 混合专家 MoE", section "细粒度专家与共享专家": a sigmoid gate decided
 * by the current token scales the shared expert's output).
 *   x [T, d] act_dtype; shared_gate [d] act_dtype (the gate's d -> 1 weight);
 *   weights [T] fp32 device.  fp32 accumulation in a fixed order. */
MOE_API moe_status_t moe_shared_gate_weights(const moe_config_t* cfg, const void* x,
                                             const void* shared_gate, float* weights,
                                             void* stream);

/* The balance-loss scalar of "10. 混合专家 MoE", section "辅助损失":
 *   *loss = alpha * E * sum_e f_e * P_e,
 *   f_e = (counts[e] + drops[e]) / sum_e' (counts[e'] + drops[e'])  (the share
 *         of assignments that chose e, dropped ones included; drops may be NULL),
 *   P_e = mean_prob[e]  (as written by moe_router_topk / the layer forward).
 * counts, drops [E] int32, mean_prob [E] fp32, loss [1] fp32, all device; one
 * small kernel on `stream`.  0 when there are no assignments. */
MOE_API moe_status_t moe_balance_loss(const moe_config_t* cfg, const int32_t* counts,
                                      const int32_t* drops, const float* mean_prob, float alpha,
                                      float* loss, void* stream);

/* The whole layer forward, stream-ordered, with no host synchronisation:
 * router -> gating/top-k -> capacity/dispatch -> gather -> grouped gate/up +
 * SwiGLU -> grouped down -> combine.
 *   y [T, d] out_dtype (required);
 *   router_bias, score_bias, ws_gate/ws_up/ws_down (all or none) may be NULL;
 *   shared_gate [d] act_dtype or NULL: when given (requires the shared
 *     expert), the shared expert's output is scaled per token by
 *     sigmoid(x_t . shared_gate) (moe_shared_gate_weights);
 *   scales: E4M3 weight scales (cfg->weight_format MOE_WEIGHTS_FP8_E4M3),
 *     else NULL;
 *   topk_idx [T, k], topk_w [T, k], counts [E], drops [E], mean_prob [E]
 *     are optional outputs (NULL = not returned); under expert choice
 *     topk_idx / topk_w must be NULL, counts[e] = C and drops[e] = 0. */
MOE_API moe_status_t moe_layer_forward(const moe_config_t* cfg, const void* x, const void* w_router,
                               const float* router_bias, const float* score_bias,
                               const void* w_gate, const void* w_up, const void* w_down,
                               const void* ws_gate, const void* ws_up, const void* ws_down,
                               const void* shared_gate, const moe_weight_scales_t* scales,
                               void* y, int32_t* topk_idx, float* topk_w,
                               int32_t* counts, int32_t* drops, float* mean_prob,
                               void* ws, size_t ws_bytes, void* stream);

/* moe_layer_forward with the token rows in host memory: enqueues, on
 * `stream`, the copy of x_host [T, d_model] (act_dtype) into the device
 * buffer x, the layer forward of x into the device buffer y, and the copy of
 * y into y_host [T, d_model] (out_dtype).  x and y are caller-owned device
 * staging buffers with the layout of moe_layer_forward; every other argument
 * is as there.  The copies are asynchronous when x_host and y_host are
 * page-locked (cudaHostAlloc or cudaHostRegister); y_host is complete once
 * `stream` has reached this call's end.  Callers that keep two batches in
 * flight on two streams (each with its own staging buffers and workspace)
 * overlap one batch's copies with the other's kernels.  Argument errors are
 * returned before anything is enqueued; a failed copy returns MOE_ERR_CUDA. */
MOE_API moe_status_t moe_layer_forward_host(const moe_config_t* cfg, const void* x_host, void* x,
                                            const void* w_router, const float* router_bias,
                                            const float* score_bias, const void* w_gate,
                                            const void* w_up, const void* w_down,
                                            const void* ws_gate, const void* ws_up,
                                            const void* ws_down, const void* shared_gate,
                                            const moe_weight_scales_t* scales, void* y,
                                            void* y_host, int32_t* topk_idx, float* topk_w,
                                            int32_t* counts, int32_t* drops, float* mean_prob,
                                            void* ws, size_t ws_bytes, void* stream);

/* Stages of moe_layer_forward, in launch order (for moe_layer_forward_profiled). */
typedef enum {
  MOE_STAGE_ROUTER = 0,    /* router logits                                  */
  MOE_STAGE_TOPK = 1,      /* gating + top-k + mean probability              */
  MOE_STAGE_DISPATCH = 2,  /* histogram, scan, scatter                       */
  MOE_STAGE_GATHER = 3,    /* grouped rows of x                              */
  MOE_STAGE_GATE_UP = 4,   /* grouped gate/up GEMM + SwiGLU                  */
  MOE_STAGE_DOWN = 5,      /* grouped down GEMM                              */
  MOE_STAGE_COMBINE = 6,   /* weighted unpermute-combine                     */
  MOE_NUM_STAGES = 7
} moe_stage_t;

/* moe_layer_forward that also records stage_events[i] (cudaEvent_t, created
 * by the caller) on `stream` right before stage i is enqueued, and
 * stage_events[MOE_NUM_STAGES] after the last one, so that the caller can
 * time each stage with cudaEventElapsedTime.  *n_launches (if not NULL)
 * receives the number of kernels this call enqueued.  Same results as
 * moe_layer_forward. */
MOE_API moe_status_t moe_layer_forward_profiled(
    const moe_config_t* cfg, const void* x, const void* w_router, const float* router_bias,
    const float* score_bias, const void* w_gate, const void* w_up, const void* w_down,
    const void* ws_gate, const void* ws_up, const void* ws_down, const void* shared_gate,
    const moe_weight_scales_t* scales, void* y, int32_t* topk_idx, float* topk_w,
    int32_t* counts, int32_t* drops,
    float* mean_prob, void* ws, size_t ws_bytes, void* stream,
    void** stage_events, int32_t* n_launches);

/* Self-test of the device-side failure detection.  Every wait inside the
 * library's tensor-core kernels is bounded; when a bound runs out the kernel
 * records MOE_ERR_TIMEOUT in the workspace status word, drains its own copies
 * in flight, frees its tensor memory and returns instead of hanging.  This
 * call launches one tiny kernel whose single bounded wait can never be
 * satisfied, with the given bound (1 ns .. 1 s), so that a caller can check
 * that moe_get_error then reports MOE_ERR_TIMEOUT and that the CUDA context
 * stays usable.  `ws` is any workspace (only its status word is used). */
MOE_API moe_status_t moe_selftest_bounded_wait(void* ws, size_t ws_bytes, uint64_t timeout_ns,
                                               void* stream);

/* Synchronises `stream`, reads and clears the workspace status word.
 * Returns MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE (or MOE_ERR_CUDA if the
 * stream itself reports an error). */
MOE_API moe_status_t moe_get_error(const void* ws, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */

// Router logits and the fused gating / top-k / renormalisation kernel.
//
// Method ("10. 混合专家 MoE：总参数与激活参数", niuwancheng.cn):
//   logits = x . W_router^T                     (block sketch, first line)
//   softmax  p_i = exp(z_i) / sum_j exp(z_j)    ("路由器怎样选专家：top-k 与两种门控")
//   sigmoid  s_i = 1 / (1 + exp(-z_i))
//   choose the k largest, renormalise over the chosen, times
//   routed_scaling_factor (2.5 for DeepSeek-V3).
// The selection compares the fp32 logits (softmax and sigmoid are increasing
// in z) with ties going to the lower expert index.
//
// DeepSeek-V3 auxiliary-loss-free routing (same page, "DeepSeek-V3 的无辅助
// 损失偏置"): with a selection-only score bias b or expert groups, the ranking
// key is s + b; a group is scored by the sum of its two largest keys, the
// best topk_group groups are kept, and the experts are chosen among them.
// The weights always use the raw scores s.
#include "internal.cuh"

#include <math.h>

namespace moe {
namespace {

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

// ---------------------------------------------------------------------------
// Router logits, SIMT tiles of 64 tokens x 64 experts, fp32 accumulation.
// ---------------------------------------------------------------------------
template <typename TIn>
__global__ void __launch_bounds__(256)
router_logits_kernel(const TIn* __restrict__ x, const TIn* __restrict__ w,
                     const float* __restrict__ bias, float* __restrict__ z,
                     int T, int E, int d) {
  __shared__ float As[32][64 + 1];
  __shared__ float Bs[32][64 + 1];
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < d; k0 += 32) {
    for (int i = threadIdx.x; i < 64 * 32; i += 256) {
      const int r = i >> 5, kk = i & 31;
      const int gk = k0 + kk;
      const int gm = m0 + r, gn = n0 + r;
      As[kk][r] = (gm < T && gk < d) ? to_f(x[(size_t)gm * d + gk]) : 0.f;
      Bs[kk][r] = (gn < E && gk < d) ? to_f(w[(size_t)gn * d + gk]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty + 16 * i;
    if (gm >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx + 16 * j;
      if (gn < E) z[(size_t)gm * E + gn] = acc[i][j] + (bias ? bias[gn] : 0.f);
    }
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// (za, ea) ranks before (zb, eb): larger logit, then lower expert index.
__device__ __forceinline__ bool ranks_before(float za, int ea, float zb, int eb) {
  return za > zb || (za == zb && ea < eb);
}

// ---------------------------------------------------------------------------
// One warp per token.  Lane l holds experts l, l+32, ... (EPL per lane).
// Block b owns tokens [b*tpb, (b+1)*tpb) so the mean-probability partial of
// each block is a fixed-order sum, and the final reduction over blocks is too.
// ---------------------------------------------------------------------------
// SCORE_KEY: rank by s + score_bias (and expert groups) instead of the logit.
template <int EPL, bool SCORE_KEY>
__global__ void __launch_bounds__(256)
topk_gate_kernel(const float* __restrict__ partials, int splits, size_t split_stride,
                 const float* __restrict__ bias, const float* __restrict__ sbias,
                 int n_group, int topk_group, float* __restrict__ logits_out, int T, int E,
                 int k, int gate, int renorm, float rsf, int tpb, int32_t* __restrict__ idx_out,
                 float* __restrict__ w_out, float* __restrict__ mp_partial) {
  __shared__ float red[8][kMaxExperts];   // logits of the chunk's tokens, then score partials
  __shared__ float keys[SCORE_KEY ? 8 : 1][SCORE_KEY ? kMaxExperts : 1];   // per-warp ranking keys
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float acc[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) acc[i] = 0.f;

  const int t_begin = blockIdx.x * tpb;
  const int t_end = min(T, t_begin + tpb);
  // With more than two split partials (a small batch), the whole block sums
  // them first; otherwise each lane adds its own experts' partials.
  const bool presum = splits > 2;
  // chunks of 8 tokens, warp w taking token t0 + w
  for (int t0 = t_begin; t0 < t_end; t0 += 8) {
    const int nt = min(8, t_end - t0);
    if (presum) {
      // the chunk's logits: the whole block sums the split partials (in split
      // order) for 8 tokens x E experts, every load independent of the others
      __syncthreads();   // red[] of the previous chunk has been read
      for (int j = threadIdx.x; j < nt * E; j += blockDim.x) {
        const int tk = j / E, e = j - tk * E;
        const float* src = partials + (size_t)(t0 + tk) * E + e;
        float pv[kMaxRouterSplits];
#pragma unroll
        for (int sp = 0; sp < kMaxRouterSplits; ++sp)
          pv[sp] = sp < splits ? src[(size_t)sp * split_stride] : 0.f;
        float v = pv[0];
#pragma unroll
        for (int sp = 1; sp < kMaxRouterSplits; ++sp)
          if (sp < splits) v += pv[sp];
        if (bias) v += bias[e];
        red[tk][e] = v;
        if (logits_out) logits_out[(size_t)(t0 + tk) * E + e] = v;
      }
      __syncthreads();
    }
    const int t = t0 + warp;
    if (warp >= nt) continue;
    float zv[EPL], sc[EPL];
    if (presum) {
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        zv[i] = e < E ? red[warp][e] : -INFINITY;
      }
    } else {
      const float* row = partials + (size_t)t * E;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
          float v = row[e];
          if (splits > 1) v += row[split_stride + e];
          if (bias) v += bias[e];
          zv[i] = v;
          if (logits_out) logits_out[(size_t)t * E + e] = v;
        } else {
          zv[i] = -INFINITY;
        }
      }
    }
    if (gate == MOE_GATE_SOFTMAX) {
      float m = -INFINITY;
#pragma unroll
      for (int i = 0; i < EPL; ++i) m = fmaxf(m, zv[i]);
      m = warp_max(m);
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        sc[i] = (lane + 32 * i < E) ? expf(zv[i] - m) : 0.f;
        s += sc[i];
      }
      s = warp_sum(s);
#pragma unroll
      for (int i = 0; i < EPL; ++i) sc[i] = sc[i] / s;
    } else {
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        sc[i] = (lane + 32 * i < E) ? 1.f / (1.f + expf(-zv[i])) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[i] += sc[i];

    // ranking value of each of this lane's experts, and the kept groups
    float rv[EPL];
    uint32_t gkeep = 0xffffffffu;
    int gsize = E;
    if (SCORE_KEY) {
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        rv[i] = e < E ? sc[i] + (sbias ? sbias[e] : 0.f) : -INFINITY;
      }
      if (n_group > 1) {
        gsize = E / n_group;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
          const int e = lane + 32 * i;
          if (e < E) keys[warp][e] = rv[i];
        }
        __syncwarp();
        // lane g scores group g: its two largest keys, added
        float gsc = -INFINITY;
        if (lane < n_group) {
          float t1 = -INFINITY, t2 = -INFINITY;
          for (int e = lane * gsize; e < (lane + 1) * gsize; ++e) {
            const float v = keys[warp][e];
            if (v > t1) {
              t2 = t1;
              t1 = v;
            } else if (v > t2) {
              t2 = v;
            }
          }
          gsc = t1 + t2;
        }
        gkeep = 0;
        for (int r = 0; r < topk_group; ++r) {
          const bool cand = lane < n_group && !((gkeep >> lane) & 1u);
          float bz = cand ? gsc : -INFINITY;
          int be = cand ? lane : 0x7fffffff;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float oz = __shfl_xor_sync(0xffffffffu, bz, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (ranks_before(oz, oe, bz, be)) {
              bz = oz;
              be = oe;
            }
          }
          gkeep |= 1u << (be & 31);
        }
        __syncwarp();   // keys[warp] is rewritten by the next token
      }
    } else {
#pragma unroll
      for (int i = 0; i < EPL; ++i) rv[i] = zv[i];
    }

    unsigned selmask = 0;
    int my_e = 0;
    float my_s = 0.f;
    for (int j = 0; j < k; ++j) {
      float bz = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        const bool allowed = !SCORE_KEY || ((gkeep >> (e / gsize)) & 1u);
        if (e < E && allowed && !((selmask >> i) & 1u) && ranks_before(rv[i], e, bz, be)) {
          bz = rv[i];
          be = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float oz = __shfl_xor_sync(0xffffffffu, bz, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ranks_before(oz, oe, bz, be)) {
          bz = oz;
          be = oe;
        }
      }
      const int owner = be & 31, slot = be >> 5;
      float s_sel = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (i == slot) s_sel = sc[i];
      s_sel = __shfl_sync(0xffffffffu, s_sel, owner);
      if (lane == owner) selmask |= 1u << slot;
      if (lane == j) {
        my_e = be;
        my_s = s_sel;
      }
    }
    float ssum = 0.f;
    for (int j = 0; j < k; ++j) ssum += __shfl_sync(0xffffffffu, my_s, j);
    if (lane < k) {
      float g = renorm ? my_s / ssum : my_s;
      g *= rsf;
      idx_out[(size_t)t * k + lane] = my_e;
      w_out[(size_t)t * k + lane] = g;
    }
  }
  if (mp_partial == nullptr) return;
  __syncthreads();   // every warp is done with the last chunk's logits
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) red[warp][e] = acc[i];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += red[w][e];
    mp_partial[(size_t)blockIdx.x * E + e] = s;
  }
}

// One step of the auxiliary-loss-free bias: b_e -= gamma * sign(E * load_e -
// sum load), load = counts (+ drops), compared in integers.  One block.
__global__ void __launch_bounds__(kMaxExperts)
score_bias_update_kernel(const int32_t* __restrict__ counts, const int32_t* __restrict__ drops,
                         int E, float gamma, float* __restrict__ bias) {
  __shared__ long long part[kMaxExperts / 32];
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  const long long load = e < E ? (long long)counts[e] + (drops ? (long long)drops[e] : 0) : 0;
  long long s = load;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) part[warp] = s;
  __syncthreads();
  long long total = 0;
  for (int w = 0; w < kMaxExperts / 32; ++w) total += part[w];
  if (e < E) {
    const long long diff = (long long)E * load - total;
    if (diff > 0) bias[e] -= gamma;
    else if (diff < 0) bias[e] += gamma;
  }
}

// Per-token weight of the shared expert, sigmoid(x_t . w) ("细粒度专家与共享
// 专家": a token-dependent sigmoid gate in front of the shared expert).  One
// warp per token, fp32 accumulation in a fixed order.
template <typename TIn>
__global__ void __launch_bounds__(256)
shared_gate_kernel(const TIn* __restrict__ x, const TIn* __restrict__ w, int T, int d,
                   float* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const TIn* row = x + (size_t)t * d;
  float acc = 0.f;
  for (int c = lane; c < d; c += 32) acc = fmaf(to_f(row[c]), to_f(w[c]), acc);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) out[t] = 1.f / (1.f + expf(-acc));
}

// alpha * N * sum_e f_e * P_e with f_e = (counts_e + drops_e) / sum of loads
// ("辅助损失").  One block, fixed-order sums.
__global__ void __launch_bounds__(kMaxExperts)
balance_loss_kernel(const int32_t* __restrict__ counts, const int32_t* __restrict__ drops,
                    const float* __restrict__ mean_prob, int E, float alpha,
                    float* __restrict__ loss) {
  __shared__ double fp[kMaxExperts];
  __shared__ long long ld[kMaxExperts];
  const int e = threadIdx.x;
  const long long load = e < E ? (long long)counts[e] + (drops ? (long long)drops[e] : 0) : 0;
  ld[e] = load;
  fp[e] = e < E ? (double)load * (double)mean_prob[e] : 0.0;
  __syncthreads();
  if (e == 0) {
    long long total = 0;
    double s = 0.0;
    for (int i = 0; i < E; ++i) {
      total += ld[i];
      s += fp[i];
    }
    *loss = total > 0 ? (float)((double)alpha * (double)E * s / (double)total) : 0.f;
  }
}

// mean_prob[e] = (sum over the top-k blocks' partials) / T.  One block per
// 32 experts: warp w adds the partials of blocks w, w + 32, ... for expert
// e0 + lane (eight loads in flight), then lane e of warp 0 adds the 32 warp
// sums in warp order, a fixed order whatever the timing.
constexpr int kFinalizeWarps = 32;
__global__ void __launch_bounds__(kFinalizeWarps * 32)
mean_prob_finalize_kernel(const float* __restrict__ mp_partial, int nblocks, int E, int T,
                          float* __restrict__ mean_prob) {
  __shared__ float ws[kFinalizeWarps][33];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + lane;
  float s = 0.f;
  if (e < E) {
    int b = warp;
    for (; b + 7 * kFinalizeWarps < nblocks; b += 8 * kFinalizeWarps) {
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = mp_partial[(size_t)(b + i * kFinalizeWarps) * E + e];
#pragma unroll
      for (int i = 0; i < 8; ++i) s += v[i];
    }
    for (; b < nblocks; b += kFinalizeWarps) s += mp_partial[(size_t)b * E + e];
  }
  ws[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && e < E) {
    float t = 0.f;
#pragma unroll 8
    for (int w = 0; w < kFinalizeWarps; ++w) t += ws[w][lane];
    mean_prob[e] = T > 0 ? t / (float)T : 0.f;
  }
}

}  // namespace

cudaError_t launch_router(const moe_config_t& c, const void* x, const void* w_router,
                          const float* bias, float* scratch, LogitsView* view, int32_t* status,
                          cudaStream_t s, LaunchCounter* lc) {
  view->partials = scratch;
  view->split_stride = (size_t)c.T * c.n_experts;
  if (c.T == 0) {
    view->splits = 1;
    view->bias = nullptr;
    return cudaSuccess;
  }
  if (c.act_dtype == MOE_BF16) {
    // tensor cores; the bias is added where the partial sums are combined
    view->splits = plan_router(c).splits;
    view->bias = bias;
    return launch_router_tc(c, x, w_router, scratch, status, s, lc);
  }
  view->splits = 1;
  view->bias = nullptr;
  dim3 grid((c.n_experts + 63) / 64, (c.T + 63) / 64);
  router_logits_kernel<float><<<grid, 256, 0, s>>>((const float*)x, (const float*)w_router, bias,
                                                   scratch, c.T, c.n_experts, c.d_model);
  count_launch(lc);
  return cudaGetLastError();
}

cudaError_t launch_mean_prob_finalize(const float* mp_partial, int nblocks, int E, int T,
                                      float* mean_prob, cudaStream_t s, LaunchCounter* lc) {
  mean_prob_finalize_kernel<<<(E + 31) / 32, kFinalizeWarps * 32, 0, s>>>(mp_partial, nblocks,
                                                                          E, T, mean_prob);
  count_launch(lc);
  return cudaGetLastError();
}

cudaError_t launch_score_bias_update(const moe_config_t& c, const int32_t* counts,
                                     const int32_t* drops, float gamma, float* bias,
                                     cudaStream_t s) {
  score_bias_update_kernel<<<1, kMaxExperts, 0, s>>>(counts, drops, c.n_experts, gamma, bias);
  return cudaGetLastError();
}

cudaError_t launch_shared_gate(const moe_config_t& c, const void* x, const void* w, float* out,
                               cudaStream_t s, LaunchCounter* lc) {
  if (c.T == 0) return cudaSuccess;
  const int blocks = (c.T + 7) / 8;
  if (c.act_dtype == MOE_BF16)
    shared_gate_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
        (const __nv_bfloat16*)x, (const __nv_bfloat16*)w, c.T, c.d_model, out);
  else
    shared_gate_kernel<float><<<blocks, 256, 0, s>>>((const float*)x, (const float*)w, c.T,
                                                     c.d_model, out);
  count_launch(lc);
  return cudaGetLastError();
}

cudaError_t launch_balance_loss(const moe_config_t& c, const int32_t* counts,
                                const int32_t* drops, const float* mean_prob, float alpha,
                                float* loss, cudaStream_t s) {
  balance_loss_kernel<<<1, kMaxExperts, 0, s>>>(counts, drops, mean_prob, c.n_experts, alpha,
                                                loss);
  return cudaGetLastError();
}

cudaError_t launch_topk(const moe_config_t& c, const LogitsView& z, const float* score_bias,
                        float* logits_out, int32_t* idx, float* w, float* mp_partial,
                        float* mean_prob, cudaStream_t s, LaunchCounter* lc) {
  const int T = c.T, E = c.n_experts;
  if (T == 0) {
    if (mean_prob) return cudaMemsetAsync(mean_prob, 0, sizeof(float) * E, s);
    return cudaSuccess;
  }
  // up to 8 tokens per block (one per warp), fewer when the batch would
  // not fill the GPU: the block sums a token's split partials with one
  // thread per expert, so a small batch takes one block per token
  int tpb = T / sm_count();
  tpb = tpb < 1 ? 1 : (tpb > 8 ? 8 : tpb);
  int nblocks = (T + tpb - 1) / tpb;
  if (nblocks > kTopkMaxBlocks) {
    nblocks = kTopkMaxBlocks;
    tpb = (T + nblocks - 1) / nblocks;
    nblocks = (T + tpb - 1) / tpb;
  }
  float* part = mean_prob ? mp_partial : nullptr;
  const bool score_key = score_bias != nullptr || c.n_group > 1;
  const int ng = c.n_group > 1 ? c.n_group : 1;
#define MOE_TOPK_LAUNCH(EPL, SK)                                                          \
  topk_gate_kernel<EPL, SK><<<nblocks, 256, 0, s>>>(                                     \
      z.partials, z.splits, z.split_stride, z.bias, score_bias, ng, c.topk_group,        \
      logits_out, T, E, c.top_k, c.gate, c.renormalize, c.routed_scaling_factor, tpb,    \
      idx, w, part)
#define MOE_TOPK_EPL(SK)                   \
  if (E <= 32) MOE_TOPK_LAUNCH(1, SK);     \
  else if (E <= 64) MOE_TOPK_LAUNCH(2, SK);  \
  else if (E <= 128) MOE_TOPK_LAUNCH(4, SK); \
  else MOE_TOPK_LAUNCH(8, SK);
  if (score_key) {
    MOE_TOPK_EPL(true)
  } else {
    MOE_TOPK_EPL(false)
  }
#undef MOE_TOPK_EPL
#undef MOE_TOPK_LAUNCH
  count_launch(lc);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess || !mean_prob) return err;
  mean_prob_finalize_kernel<<<(E + 31) / 32, kFinalizeWarps * 32, 0, s>>>(mp_partial, nblocks,
                                                                          E, T, mean_prob);
  count_launch(lc);
  return cudaGetLastError();
}

}  // namespace moe

// Expert-choice routing: each expert takes a fixed number of the tokens it
// scores highest (the amazingdata.cn article on MoE routing, paragraph on
// expert choice; the load is balanced by construction and a token may be
// taken by no expert).
//
//   scores   s[t, e] = softmax_e(z[t, :]) or sigmoid(z[t, e])  (fp32)
//   select   expert e takes the C tokens with the largest s[t, e], ties to
//            the lower token, listed in ascending token order
//   combine  y_t = sum over the experts e that took t, in ascending e, of
//            s[t, e] * E_e(x_t)   (+ the shared expert)
//
// Kernels:
//   ec_scores_kernel   one warp per token; writes the scores transposed
//                      [E, T] and per-block partial sums for the mean
//                      probability (fixed order);
//   ec_select_kernel   one block per expert: the column's scores become
//                      order-preserving 32-bit keys in shared memory, four
//                      8-bit radix passes find the C-th largest key, and
//                      block prefix sums over token order emit the chosen
//                      tokens ascending (exact, deterministic, no sort);
//   ec_combine_kernel  one block per token: the [T, E] row map that the
//                      selection fills (-1 where expert e did not take t)
//                      gives the token's rows, summed in ascending expert
//                      order.
#include "internal.cuh"

#include <math.h>

namespace moe {
namespace {

constexpr int kSelThreads = 1024;

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Block per tpb tokens (8 warps), lane l holds experts l, l+32, ...
template <int EPL>
__global__ void __launch_bounds__(256)
ec_scores_kernel(const float* __restrict__ partials, int splits, size_t split_stride,
                 const float* __restrict__ bias, int T, int E, int gate, int tpb,
                 float* __restrict__ scores_t, float* __restrict__ mp_partial) {
  __shared__ float red[8][kMaxExperts];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float acc[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) acc[i] = 0.f;
  const int t_begin = blockIdx.x * tpb;
  const int t_end = min(T, t_begin + tpb);
  for (int t = t_begin + warp; t < t_end; t += 8) {
    const float* row = partials + (size_t)t * E;
    float zv[EPL], sc[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        float v = row[e];
        for (int sp = 1; sp < splits; ++sp) v += row[(size_t)sp * split_stride + e];
        if (bias) v += bias[e];
        zv[i] = v;
      } else {
        zv[i] = -INFINITY;
      }
    }
    if (gate == MOE_GATE_SOFTMAX) {
      float m = -INFINITY;
#pragma unroll
      for (int i = 0; i < EPL; ++i) m = fmaxf(m, zv[i]);
      m = warp_max_f(m);
      float ssum = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        sc[i] = (lane + 32 * i < E) ? expf(zv[i] - m) : 0.f;
        ssum += sc[i];
      }
      ssum = warp_sum_f(ssum);
#pragma unroll
      for (int i = 0; i < EPL; ++i) sc[i] = sc[i] / ssum;
    } else {
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        sc[i] = (lane + 32 * i < E) ? 1.f / (1.f + expf(-zv[i])) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        scores_t[(size_t)e * T + t] = sc[i];
        acc[i] += sc[i];
      }
    }
  }
  if (mp_partial == nullptr) return;
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

// Exclusive prefix sum over the block (1024 threads) in thread order; also
// returns the total.
__device__ __forceinline__ int block_scan(int v, int* wsum, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    wsum[lane] = w;   // inclusive over warps
  }
  __syncthreads();
  total = wsum[31];
  const int before = (warp > 0 ? wsum[warp - 1] : 0) + x - v;
  __syncthreads();
  return before;
}

// fp32 -> 32-bit key whose unsigned order is the float order.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__global__ void __launch_bounds__(kSelThreads)
ec_select_kernel(const float* __restrict__ scores_t, int T, int E, int C,
                 int32_t* __restrict__ tokens, float* __restrict__ weights,
                 int32_t* __restrict__ rowmap, int32_t* __restrict__ offsets,
                 int32_t* __restrict__ counts, int32_t* __restrict__ drops) {
  extern __shared__ uint32_t keys[];   // [T]
  __shared__ int hist[256];
  __shared__ int wsum[32];
  __shared__ uint32_t s_prefix;
  __shared__ int s_rank;
  const int e = blockIdx.x, tid = threadIdx.x;
  if (tid == 0) {
    offsets[e] = e * C;
    counts[e] = C;
    drops[e] = 0;
    if (e == 0) offsets[E] = E * C;
  }
  if (C == 0) return;
  const float* col = scores_t + (size_t)e * T;
  for (int t = tid; t < T; t += kSelThreads) keys[t] = order_key(col[t]);
  if (tid == 0) {
    s_prefix = 0;
    s_rank = C;
  }
  __syncthreads();
  // radix select of the C-th largest key, 8 bits at a time from the top
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    const uint32_t hi_mask = pass == 0 ? 0u : (0xFFFFFFFFu << (shift + 8));
    for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix;
    for (int t = tid; t < T; t += kSelThreads) {
      const uint32_t k = keys[t];
      if ((k & hi_mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1);
    }
    __syncthreads();
    if (tid == 0) {
      int r = s_rank, above = 0, dgt = 255;
      for (; dgt > 0; --dgt) {
        if (above + hist[dgt] >= r) break;
        above += hist[dgt];
      }
      s_prefix = prefix | ((uint32_t)dgt << shift);
      s_rank = r - above;
    }
    __syncthreads();
  }
  const uint32_t theta = s_prefix;   // the C-th largest key
  const int take_eq = s_rank;        // keys equal to theta to take, lowest tokens first
  // each thread scans a contiguous run of tokens so that prefix sums follow
  // token order
  const int run = (T + kSelThreads - 1) / kSelThreads;
  const int t0 = min(T, tid * run), t1 = min(T, t0 + run);
  int n_eq = 0;
  for (int t = t0; t < t1; ++t) n_eq += keys[t] == theta ? 1 : 0;
  int tot;
  int eq_before = block_scan(n_eq, wsum, tot);
  int n_sel = 0;
  {
    int q = eq_before;
    for (int t = t0; t < t1; ++t) {
      const uint32_t k = keys[t];
      if (k > theta) ++n_sel;
      else if (k == theta) n_sel += (q++ < take_eq) ? 1 : 0;
    }
  }
  int pos = block_scan(n_sel, wsum, tot);
  {
    int q = eq_before;
    for (int t = t0; t < t1; ++t) {
      const uint32_t k = keys[t];
      bool sel = k > theta;
      if (k == theta) sel = (q++ < take_eq);
      if (sel && pos < C) {
        tokens[(size_t)e * C + pos] = t;
        weights[(size_t)e * C + pos] = col[t];
        if (rowmap) rowmap[(size_t)t * E + e] = e * C + pos;
        ++pos;
      }
    }
  }
}

// One block per token (grid-stride): the token's rows from the row map, summed
// in ascending expert order; one write of y.
template <typename TOut>
__global__ void __launch_bounds__(256)
ec_combine_kernel(const float4* __restrict__ y_perm, const int32_t* __restrict__ rowmap,
                  const float* __restrict__ weights, const float4* __restrict__ y_shared,
                  const float* __restrict__ shared_w, TOut* __restrict__ y, int T, int E, int R,
                  int d, int32_t* status) {
  __shared__ int s_row[kMaxExperts];
  __shared__ float s_g[kMaxExperts];
  __shared__ int s_n;
  const int d4 = d >> 2;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    if (threadIdx.x == 0) s_n = 0;
    __syncthreads();
    // compact the hits in expert order (a warp ballot per 32 experts)
    for (int e0 = 0; e0 < E; e0 += 32) {
      if (threadIdx.x < 32) {
        const int e = e0 + threadIdx.x;
        int r = e < E ? rowmap[(size_t)t * E + e] : -1;
        if (r >= R) {
          record_error(status, kDevBadIndex);
          r = -1;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, r >= 0);
        const int at = s_n + __popc(hit & ((1u << threadIdx.x) - 1u));
        if (r >= 0) {
          s_row[at] = r;
          s_g[at] = weights[r];
        }
        __syncwarp();
        if (threadIdx.x == 0) s_n += __popc(hit);
        __syncwarp();
      }
    }
    __syncthreads();
    const int n = s_n;
    for (int v = threadIdx.x; v < d4; v += blockDim.x) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j = 0; j < n; ++j) {
        const float g = s_g[j];
        const float4 yv = __ldg(y_perm + (size_t)s_row[j] * d4 + v);
        acc.x = fmaf(g, yv.x, acc.x);
        acc.y = fmaf(g, yv.y, acc.y);
        acc.z = fmaf(g, yv.z, acc.z);
        acc.w = fmaf(g, yv.w, acc.w);
      }
      if (y_shared) {
        const float4 sv = __ldg(y_shared + (size_t)t * d4 + v);
        const float ws = shared_w ? __ldg(shared_w + t) : 1.f;
        acc.x = fmaf(ws, sv.x, acc.x);
        acc.y = fmaf(ws, sv.y, acc.y);
        acc.z = fmaf(ws, sv.z, acc.z);
        acc.w = fmaf(ws, sv.w, acc.w);
      }
      if (sizeof(TOut) == 4) {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(y) + (size_t)t * d + 4 * v) = acc;
      } else {
        __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x, acc.y);
        __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&lo2);
        u.y = *reinterpret_cast<uint32_t*>(&hi2);
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(y) + (size_t)t * d + 4 * v) = u;
      }
    }
    __syncthreads();
  }
}

int sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      n = 148;
  }
  return n;
}

}  // namespace

cudaError_t launch_ec_route(const moe_config_t& c, const LogitsView& z, float* scores_t,
                            float* mp_partial, float* mean_prob, int32_t* tokens, float* weights,
                            int32_t* rowmap, int32_t* offsets, int32_t* counts, int32_t* drops,
                            cudaStream_t s, LaunchCounter* lc) {
  const int T = c.T, E = c.n_experts, C = ec_capacity(c);
  int nblocks = (T + 7) / 8;
  if (nblocks > kTopkMaxBlocks) nblocks = kTopkMaxBlocks;
  if (nblocks < 1) nblocks = 1;
  const int tpb = (T + nblocks - 1) / nblocks;
  if (T > 0) {
    nblocks = (T + tpb - 1) / tpb;
    float* part = mean_prob ? mp_partial : nullptr;
#define MOE_EC_SCORES(EPL)                                                                   \
  ec_scores_kernel<EPL><<<nblocks, 256, 0, s>>>(z.partials, z.splits, z.split_stride, z.bias, \
                                                T, E, c.gate, tpb, scores_t, part)
    if (E <= 32) MOE_EC_SCORES(1);
    else if (E <= 64) MOE_EC_SCORES(2);
    else if (E <= 128) MOE_EC_SCORES(4);
    else MOE_EC_SCORES(8);
#undef MOE_EC_SCORES
    count_launch(lc);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  static cudaError_t attr = cudaFuncSetAttribute(
      ec_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kEcMaxTokens * 4);
  if (attr != cudaSuccess) return attr;
  if (rowmap && T > 0) {
    cudaError_t err = cudaMemsetAsync(rowmap, 0xff, sizeof(int32_t) * (size_t)T * E, s);
    if (err != cudaSuccess) return err;
  }
  ec_select_kernel<<<E, kSelThreads, (size_t)(T > 0 ? T : 1) * 4, s>>>(
      scores_t, T, E, C, tokens, weights, rowmap, offsets, counts, drops);
  count_launch(lc);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (mean_prob) {
    if (T == 0) return cudaMemsetAsync(mean_prob, 0, sizeof(float) * E, s);
    return launch_mean_prob_finalize(mp_partial, nblocks, E, T, mean_prob, s, lc);
  }
  return cudaSuccess;
}

cudaError_t launch_ec_combine(const moe_config_t& c, const float* y_perm, const int32_t* rowmap,
                              const float* weights, const float* y_shared, const float* shared_w,
                              void* y, int32_t* status, cudaStream_t s, LaunchCounter* lc) {
  const int T = c.T;
  if (T == 0) return cudaSuccess;
  int blocks = T;
  if (blocks > sms() * 16) blocks = sms() * 16;
  const int R = (int)grouped_rows(c);
  if (c.out_dtype == MOE_BF16)
    ec_combine_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
        (const float4*)y_perm, rowmap, weights, (const float4*)y_shared, shared_w,
        (__nv_bfloat16*)y, T, c.n_experts, R, c.d_model, status);
  else
    ec_combine_kernel<float><<<blocks, 256, 0, s>>>((const float4*)y_perm, rowmap, weights,
                                                    (const float4*)y_shared, shared_w, (float*)y,
                                                    T, c.n_experts, R, c.d_model, status);
  count_launch(lc);
  return cudaGetLastError();
}

}  // namespace moe

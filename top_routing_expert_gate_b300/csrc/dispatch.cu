// Capacity + dispatch (histogram, scan, stable scatter), row gather, and the
// weighted unpermute-combine.
//
// Method ("10. 混合专家 MoE：总参数与激活参数", niuwancheng.cn):
//   - the block sketch groups each expert's (token, slot) pairs with
//     `(idx == e).nonzero` and runs the expert on those rows; the text after
//     it says real implementations gather each expert's tokens into one
//     grouped GEMM ("把一个大 FFN 换成一组小 FFN");
//   - capacity = tokens per batch / experts x capacity factor; tokens beyond
//     it skip the expert ("负载不均：路由坍缩与丢 token");
//   - y_t = sum_{i in TopK} g_{t,i} E_i(x_t) ("MoE为什么只激活一部分专家",
//     hi-bin.com, "Router 怎样给 Token 选专家").
//
// Determinism: the histogram only counts, and the slot of assignment a is
// computed from counts of lower assignment ids (block prefix + warp prefix +
// lane rank), so every output is a pure function of topk_idx.
#include "internal.cuh"

namespace moe {
namespace {

constexpr int kRounds = kDispatchChunk / kDispatchThreads;

__device__ __forceinline__ int load_expert(const int32_t* idx, int a, int A, int E,
                                           int32_t* status) {
  if (a >= A) return -1;
  const int e = idx[a];
  if (e < 0 || e >= E) {
    record_error(status, kDevBadIndex);
    return -1;
  }
  return e;
}

// Per-block expert histogram over assignments [b*chunk, (b+1)*chunk).
__global__ void __launch_bounds__(kDispatchThreads)
dispatch_hist_kernel(const int32_t* __restrict__ idx, int A, int E,
                     int32_t* __restrict__ block_hist, int32_t* status) {
  __shared__ int hist[kMaxExperts];
  const int tid = threadIdx.x, lane = tid & 31;
  for (int e = tid; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int a0 = blockIdx.x * kDispatchChunk;
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int e = load_expert(idx, a0 + r * kDispatchThreads + tid, A, E, status);
    // warp-aggregated increment: one shared atomic per distinct expert in the warp
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[e], __popc(peers));
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) block_hist[(size_t)blockIdx.x * E + e] = hist[e];
}

// Single block: per-expert running sums over blocks, capacity cut, offsets.
__global__ void dispatch_scan_kernel(const int32_t* __restrict__ block_hist, int nb, int E,
                                     int capacity, int32_t* __restrict__ block_base,
                                     int32_t* __restrict__ counts, int32_t* __restrict__ drops,
                                     int32_t* __restrict__ offsets) {
  __shared__ int kept[kMaxExperts];
  const int e = threadIdx.x;
  if (e < E) {
    int run = 0;
    for (int b = 0; b < nb; ++b) {
      block_base[(size_t)b * E + e] = run;
      run += block_hist[(size_t)b * E + e];
    }
    const int kp = capacity >= 0 ? min(run, capacity) : run;
    counts[e] = kp;
    drops[e] = run - kp;
    kept[e] = kp;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int s = 0;
    for (int i = 0; i < E; ++i) {
      offsets[i] = s;
      s += kept[i];
    }
    offsets[E] = s;
  }
}

// Stable scatter of one chunk of assignments: slot(a) = #{a' < a : idx[a'] ==
// idx[a]}, the chunk's running slot counts starting at run[] (shared, updated),
// off[] the experts' first rows.
__device__ __forceinline__ void scatter_chunk(const int32_t* __restrict__ idx, int A, int E,
                                              int capacity, int a0, int (*wc)[kMaxExperts],
                                              int* run, const int* off, int32_t* __restrict__ perm,
                                              int32_t* __restrict__ row_of,
                                              uint8_t* __restrict__ drop_mask) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int r = 0; r < kRounds; ++r) {
    if (a0 + r * kDispatchThreads >= A) break;   // the same for the whole block
    const int a = a0 + r * kDispatchThreads + tid;
    const int e = load_expert(idx, a, A, E, nullptr);
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int lane_rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && lane == __ffs(peers) - 1) wc[warp][e] = __popc(peers);
    __syncthreads();
    for (int ee = tid; ee < E; ee += blockDim.x) {
      int s = run[ee];
#pragma unroll 8
      for (int w = 0; w < 32; ++w) {
        const int cnt = wc[w][ee];
        wc[w][ee] = s;
        s += cnt;
      }
      run[ee] = s;
    }
    __syncthreads();
    if (a < A) {
      if (e >= 0) {
        const int slot = wc[warp][e] + lane_rank;
        if (capacity < 0 || slot < capacity) {
          const int rr = off[e] + slot;
          perm[rr] = a;
          if (row_of) row_of[a] = rr;
          drop_mask[a] = 0;
        } else {
          drop_mask[a] = 1;
          if (row_of) row_of[a] = -1;
        }
      } else {
        drop_mask[a] = 1;
        if (row_of) row_of[a] = -1;
      }
    }
    __syncthreads();
    for (int i = tid; i < 32 * E; i += blockDim.x) wc[i / E][i % E] = 0;
    __syncthreads();
  }
}

// Stable scatter, one block per chunk, after the histogram and scan kernels.
__global__ void __launch_bounds__(kDispatchThreads)
dispatch_scatter_kernel(const int32_t* __restrict__ idx, int A, int E, int capacity,
                        const int32_t* __restrict__ block_base,
                        const int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                        int32_t* __restrict__ row_of, uint8_t* __restrict__ drop_mask) {
  __shared__ int wc[32][kMaxExperts];   // per-warp counts, then prefixes
  __shared__ int run[kMaxExperts];      // slots taken so far per expert
  __shared__ int off[kMaxExperts];
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += blockDim.x) {
    run[e] = block_base[(size_t)blockIdx.x * E + e];
    off[e] = offsets[e];
  }
  for (int i = tid; i < 32 * kMaxExperts; i += blockDim.x) (&wc[0][0])[i] = 0;
  __syncthreads();
  scatter_chunk(idx, A, E, capacity, blockIdx.x * kDispatchChunk, wc, run, off, perm, row_of,
                drop_mask);
}

// The whole dispatch of at most one chunk of assignments in one block:
// histogram, capacity cut, offsets, scatter (the three kernels' steps).
__global__ void __launch_bounds__(kDispatchThreads)
dispatch_small_kernel(const int32_t* __restrict__ idx, int A, int E, int capacity,
                      int32_t* __restrict__ counts, int32_t* __restrict__ drops,
                      int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                      int32_t* __restrict__ row_of, uint8_t* __restrict__ drop_mask,
                      int32_t* status) {
  __shared__ int wc[32][kMaxExperts];
  __shared__ int run[kMaxExperts];
  __shared__ int off[kMaxExperts];   // histogram, then kept counts, then first rows
  const int tid = threadIdx.x, lane = tid & 31;
  for (int e = tid; e < E; e += blockDim.x) {
    off[e] = 0;
    run[e] = 0;
  }
  for (int i = tid; i < 32 * kMaxExperts; i += blockDim.x) (&wc[0][0])[i] = 0;
  __syncthreads();
  for (int r = 0; r < kRounds && r * kDispatchThreads < A; ++r) {
    const int e = load_expert(idx, r * kDispatchThreads + tid, A, E, status);
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) atomicAdd(&off[e], __popc(peers));
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    const int load = off[e];
    const int kp = capacity >= 0 ? min(load, capacity) : load;
    counts[e] = kp;
    drops[e] = load - kp;
    off[e] = kp;
  }
  __syncthreads();
  if (tid < 32) {
    // exclusive prefix of the kept counts: lane l sums experts
    // [l*per, (l+1)*per), a warp scan gives each lane its start
    constexpr int per = (kMaxExperts + 31) / 32;
    int loc[per];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      loc[i] = e < E ? off[e] : 0;
      sum += loc[i];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run_e = incl - sum;
#pragma unroll
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) {
        off[e] = run_e;
        offsets[e] = run_e;
      }
      run_e += loc[i];
    }
    if (lane == 31) offsets[E] = incl;
  }
  __syncthreads();
  scatter_chunk(idx, A, E, capacity, 0, wc, run, off, perm, row_of, drop_mask);
}

// One warp per grouped row, 16-byte vectors; row r holds token perm[r] / k.
// Each lane keeps eight 16-byte loads in flight before storing them, so a
// warp moves 4 KB of a row per round trip to memory.
__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ perm,
                   const int32_t* __restrict__ offsets, int E, int k, int T, int rows_cap,
                   int row_vec, uint4* __restrict__ x_perm, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  int n = offsets[E];
  if (n < 0 || n > rows_cap) {
    if (blockIdx.x == 0 && threadIdx.x == 0) record_error(status, kDevBadIndex);
    n = n < 0 ? 0 : rows_cap;
  }
  for (int r = blockIdx.x * warps + (threadIdx.x >> 5); r < n; r += gridDim.x * warps) {
    const int a = perm[r];
    const int t = a / k;
    if (a < 0 || t >= T) {
      if (lane == 0) record_error(status, kDevBadIndex);
      continue;
    }
    const uint4* src = x + (size_t)t * row_vec;
    uint4* dst = x_perm + (size_t)r * row_vec;
    for (int v0 = lane; v0 < row_vec; v0 += 32 * 8) {
      uint4 buf[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (v0 + 32 * i < row_vec) buf[i] = __ldg(src + v0 + 32 * i);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (v0 + 32 * i < row_vec) dst[v0 + 32 * i] = buf[i];
    }
  }
}

__global__ void invert_perm_kernel(const int32_t* __restrict__ perm,
                                   const int32_t* __restrict__ offsets, int E, int A,
                                   int32_t* __restrict__ row_of, int32_t* status) {
  int n = offsets[E];
  if (n < 0 || n > A) {
    if (blockIdx.x == 0 && threadIdx.x == 0) record_error(status, kDevBadIndex);
    n = n < 0 ? 0 : A;
  }
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < n; r += gridDim.x * blockDim.x) {
    const int a = perm[r];
    if (a < 0 || a >= A) {
      record_error(status, kDevBadIndex);
      continue;
    }
    row_of[a] = r;
  }
}

__device__ __forceinline__ void store4(float* y, float4 v) { *(float4*)y = v; }
__device__ __forceinline__ void store4(__nv_bfloat16* y, float4 v) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *(uint32_t*)&lo;
  u.y = *(uint32_t*)&hi;
  *(uint2*)y = u;
}

// One block per (token, span of the row's four-column vectors), grid-stride:
// a large batch takes whole rows (span = the row), a small one splits each row
// into spans of 256 vectors so that it still spreads over the GPU.  fp32
// accumulation in ascending j, then the shared expert (times its per-token
// gate when given); one write of y.
constexpr int kCombineVecs = 256;
template <typename TOut>
__global__ void __launch_bounds__(kCombineVecs)
combine_kernel(const float4* __restrict__ y_perm, const float* __restrict__ topk_w,
               const int32_t* __restrict__ row_of, const uint8_t* __restrict__ drop_mask,
               const float4* __restrict__ y_shared, const float* __restrict__ shared_w,
               TOut* __restrict__ y, int T, int k, int d, int A, int nch, int32_t* status) {
  __shared__ int s_row[kMaxTopK];
  __shared__ float s_g[kMaxTopK];
  const int d4 = d >> 2;
  const int span = (d4 + nch - 1) / nch;
  for (int w = blockIdx.x; w < T * nch; w += gridDim.x) {
    const int t = w / nch;
    const int v0 = (w - t * nch) * span;
    const int v1 = min(d4, v0 + span);
    if (threadIdx.x < k) {
      const int a = t * k + threadIdx.x;
      int r = -1;
      if (!drop_mask[a]) {
        r = row_of[a];
        if (r < 0 || r >= A) {
          record_error(status, kDevBadIndex);
          r = -1;
        }
      }
      s_row[threadIdx.x] = r;
      s_g[threadIdx.x] = topk_w[a];
    }
    __syncthreads();
    for (int v = v0 + (int)threadIdx.x; v < v1; v += blockDim.x) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j = 0; j < k; ++j) {
        const int r = s_row[j];
        if (r < 0) continue;
        const float g = s_g[j];
        const float4 yv = __ldg(y_perm + (size_t)r * d4 + v);
        acc.x = fmaf(g, yv.x, acc.x);
        acc.y = fmaf(g, yv.y, acc.y);
        acc.z = fmaf(g, yv.z, acc.z);
        acc.w = fmaf(g, yv.w, acc.w);
      }
      if (y_shared) {
        const float4 sv = __ldg(y_shared + (size_t)t * d4 + v);
        if (shared_w) {
          const float ws = __ldg(shared_w + t);
          acc.x = fmaf(ws, sv.x, acc.x);
          acc.y = fmaf(ws, sv.y, acc.y);
          acc.z = fmaf(ws, sv.z, acc.z);
          acc.w = fmaf(ws, sv.w, acc.w);
        } else {
          acc.x += sv.x;
          acc.y += sv.y;
          acc.z += sv.z;
          acc.w += sv.w;
        }
      }
      store4(y + (size_t)t * d + 4 * v, acc);
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_dispatch(const moe_config_t& c, const int32_t* idx, int32_t* block_hist,
                            int32_t* block_base, int32_t* counts, int32_t* drops,
                            int32_t* offsets, int32_t* perm, int32_t* row_of,
                            uint8_t* drop_mask, int32_t* status, cudaStream_t s,
                            LaunchCounter* lc) {
  const int A = c.T * c.top_k, E = c.n_experts;
  const int nb = (A + kDispatchChunk - 1) / kDispatchChunk;
  if (nb == 1) {
    // one chunk: the three steps in one block
    dispatch_small_kernel<<<1, kDispatchThreads, 0, s>>>(idx, A, E, c.capacity, counts, drops,
                                                         offsets, perm, row_of, drop_mask,
                                                         status);
    count_launch(lc);
    return cudaGetLastError();
  }
  if (nb > 0) {
    dispatch_hist_kernel<<<nb, kDispatchThreads, 0, s>>>(idx, A, E, block_hist, status);
    count_launch(lc);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  dispatch_scan_kernel<<<1, kMaxExperts, 0, s>>>(block_hist, nb, E, c.capacity, block_base,
                                                 counts, drops, offsets);
  count_launch(lc);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess || nb == 0) return err;
  dispatch_scatter_kernel<<<nb, kDispatchThreads, 0, s>>>(idx, A, E, c.capacity, block_base,
                                                          offsets, perm, row_of, drop_mask);
  count_launch(lc);
  return cudaGetLastError();
}

cudaError_t launch_gather(const moe_config_t& c, const void* x, const int32_t* perm,
                          const int32_t* offsets, void* x_perm, int32_t* status,
                          cudaStream_t s, LaunchCounter* lc, int div) {
  const int A = (int)grouped_rows(c);
  if (A == 0 || c.T == 0) return cudaSuccess;
  if (div <= 0) div = c.routing == MOE_ROUTE_EXPERT_CHOICE ? 1 : c.top_k;
  const int row_vec = (int)(c.d_model * act_bytes(c) / 16);
  int blocks = (A + 7) / 8;
  const int cap = sm_count() * 8;
  if (blocks > cap) blocks = cap;
  gather_rows_kernel<<<blocks, 256, 0, s>>>((const uint4*)x, perm, offsets, c.n_experts, div,
                                            c.T, A, row_vec, (uint4*)x_perm, status);
  count_launch(lc);
  return cudaGetLastError();
}

cudaError_t launch_invert_perm(const moe_config_t& c, const int32_t* perm,
                               const int32_t* offsets, int32_t* row_of, int32_t* status,
                               cudaStream_t s, LaunchCounter* lc) {
  const int A = c.T * c.top_k;
  if (A == 0) return cudaSuccess;
  cudaError_t err = cudaMemsetAsync(row_of, 0xff, sizeof(int32_t) * (size_t)A, s);
  if (err != cudaSuccess) return err;
  int blocks = (A + 255) / 256;
  if (blocks > sm_count() * 4) blocks = sm_count() * 4;
  invert_perm_kernel<<<blocks, 256, 0, s>>>(perm, offsets, c.n_experts, A, row_of, status);
  count_launch(lc);
  return cudaGetLastError();
}

cudaError_t launch_combine(const moe_config_t& c, const float* y_perm, const float* topk_w,
                           const int32_t* row_of, const uint8_t* drop_mask,
                           const float* y_shared, const float* shared_w, void* y,
                           int32_t* status, cudaStream_t s, LaunchCounter* lc) {
  const int T = c.T;
  if (T == 0) return cudaSuccess;
  // split rows only when the batch alone would not fill the GPU
  const int nch = T < 2 * sm_count() ? (c.d_model / 4 + kCombineVecs - 1) / kCombineVecs : 1;
  long long blocks = (long long)T * nch;
  if (blocks > sm_count() * 16) blocks = sm_count() * 16;
  const int A = T * c.top_k;
  if (c.out_dtype == MOE_BF16)
    combine_kernel<__nv_bfloat16><<<(int)blocks, kCombineVecs, 0, s>>>(
        (const float4*)y_perm, topk_w, row_of, drop_mask, (const float4*)y_shared, shared_w,
        (__nv_bfloat16*)y, T, c.top_k, c.d_model, A, nch, status);
  else
    combine_kernel<float><<<(int)blocks, kCombineVecs, 0, s>>>(
        (const float4*)y_perm, topk_w, row_of, drop_mask, (const float4*)y_shared, shared_w,
        (float*)y, T, c.top_k, c.d_model, A, nch, status);
  count_launch(lc);
  return cudaGetLastError();
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Dispatch without a caller-provided workspace.
//
// The two per-block tables the dispatch kernels need (histogram and running
// base, each [blocks, E] int32) live in one fixed device array compiled into
// this library instead of in the caller's workspace.  Every GPU that loads
// the library holds this array (64 KiB) until the process exits.  Host code
// cannot use the array's name as a device address, so every call looks the
// address up on the current device with cudaGetSymbolAddress (a host-side
// lookup) and passes it to the kernels like any other pointer.  Looking it up
// each time, rather than caching it, keeps it right after a cudaDeviceReset,
// which reloads the library's device code and may move the array.
// ---------------------------------------------------------------------------
namespace moe {
namespace {

constexpr int kStaticDispatchBlocks = 32;   // 32 x 4096 = 131072 assignments
constexpr int kStaticScratchInts = 2 * kStaticDispatchBlocks * kMaxExperts;

static __device__ __align__(256) int32_t g_dispatch_scratch[kStaticScratchInts];

// Device address of g_dispatch_scratch on the current device.
cudaError_t static_scratch(int32_t** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
  if (e != cudaSuccess) return e;
  *out = static_cast<int32_t*>(p);
  return cudaSuccess;
}

bool aligned16_ptr(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_dispatch_no_workspace(const moe_config_t* cfg,
                                                  const int32_t* topk_idx, int32_t* counts,
                                                  int32_t* drops, int32_t* offsets,
                                                  int32_t* perm, uint8_t* drop_mask,
                                                  void* stream) {
  using namespace moe;
  // the configuration rules of moe_dispatch, then this entry point's limit
  const moe_status_t st = validate_config(cfg);
  if (st != MOE_OK) return st;
  const moe_config_t& c = *cfg;
  if (c.routing != MOE_ROUTE_TOKEN_CHOICE) return MOE_ERR_INVALID_ARG;
  const long long A = (long long)c.T * c.top_k;
  if (A > (long long)kStaticDispatchBlocks * kDispatchChunk) return MOE_ERR_UNSUPPORTED;
  if (!counts || !drops || !offsets || !aligned16_ptr(counts) || !aligned16_ptr(drops) ||
      !aligned16_ptr(offsets))
    return MOE_ERR_INVALID_ARG;
  if (A > 0 && (!topk_idx || !perm || !drop_mask || !aligned16_ptr(topk_idx) ||
                !aligned16_ptr(perm) || !aligned16_ptr(drop_mask)))
    return MOE_ERR_INVALID_ARG;
  int32_t* scratch = nullptr;
  if (static_scratch(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  // Both tables are fully written before they are read (histogram, then
  // running base), so nothing has to be cleared between calls.
  int32_t* block_hist = scratch;
  int32_t* block_base = scratch + kStaticDispatchBlocks * kMaxExperts;
  const cudaError_t e = launch_dispatch(c, topk_idx, block_hist, block_base, counts, drops,
                                        offsets, perm, nullptr, drop_mask, nullptr,
                                        (cudaStream_t)stream);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

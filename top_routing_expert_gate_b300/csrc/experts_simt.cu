// Grouped SwiGLU experts with CUDA-core (SIMT) tiles.  This is the fp32
// activation path (the tiny fp32 layer); bf16 layers use the tcgen05 tensor
// core kernels in experts_tc.cu.
//
// Expert e ("10. 混合专家 MoE：总参数与激活参数", niuwancheng.cn,
// "把一个大 FFN 换成一组小 FFN"): gate and up are d -> F projections, SwiGLU
// activation SiLU(gate) * up, down is F -> d.
#include "internal.cuh"

namespace moe {
namespace {

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ void from_f(float v, float* p) { *p = v; }
__device__ __forceinline__ void from_f(float v, __nv_bfloat16* p) { *p = __float2bfloat16_rn(v); }

struct SimtArgs {
  const void* a_routed;    // [A, K] rows grouped by expert
  const void* a_shared;    // [T, K_s]
  const int32_t* offsets;  // [E + 1]
  const void* b0;          // routed gate (SWIGLU) or down  [E, N, K]
  const void* b1;          // routed up (SWIGLU)
  const void* bs0;         // shared gate / down [N_s, K_s]
  const void* bs1;         // shared up
  void* out_routed;        // [A, N]
  void* out_shared;        // [T, N_s]
  int E, T, rows_cap, K, N, K_s, N_s;   // rows_cap: rows of the grouped buffers
  int has_shared;
};

// 64 x 64 output tile, 256 threads, 4 x 4 outputs per thread (strided by 16
// so shared-memory reads are conflict-free), K step 32.
template <typename TIn, bool SWIGLU>
__global__ void __launch_bounds__(256) experts_simt_kernel(SimtArgs p) {
  __shared__ float As[32][64 + 1];
  __shared__ float Bs[32][64 + 1];
  __shared__ float Us[SWIGLU ? 32 : 1][64 + 1];
  const int g = blockIdx.z;
  const bool shared = (g == p.E);
  if (shared && !p.has_shared) return;
  int rows, row0, K, N;
  const TIn *A, *B0, *B1;
  if (!shared) {
    // clamp caller-provided offsets to the grouped buffer [0, A)
    const int n_assign = p.rows_cap;
    row0 = min(max(p.offsets[g], 0), n_assign);
    rows = min(max(p.offsets[g + 1], row0), n_assign) - row0;
    K = p.K;
    N = p.N;
    A = (const TIn*)p.a_routed + (size_t)row0 * K;
    B0 = (const TIn*)p.b0 + (size_t)g * N * K;
    B1 = SWIGLU ? (const TIn*)p.b1 + (size_t)g * N * K : nullptr;
  } else {
    row0 = 0;
    rows = p.T;
    K = p.K_s;
    N = p.N_s;
    A = (const TIn*)p.a_shared;
    B0 = (const TIn*)p.bs0;
    B1 = SWIGLU ? (const TIn*)p.bs1 : nullptr;
  }
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  if (m0 >= rows || n0 >= N) return;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4], acu[SWIGLU ? 4 : 1][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[i][j] = 0.f;
      if (SWIGLU) acu[SWIGLU ? i : 0][j] = 0.f;
    }
  for (int k0 = 0; k0 < K; k0 += 32) {
    for (int i = threadIdx.x; i < 64 * 32; i += 256) {
      const int r = i >> 5, kk = i & 31, gk = k0 + kk;
      const bool kin = gk < K;
      As[kk][r] = (m0 + r < rows && kin) ? to_f(A[(size_t)(m0 + r) * K + gk]) : 0.f;
      Bs[kk][r] = (n0 + r < N && kin) ? to_f(B0[(size_t)(n0 + r) * K + gk]) : 0.f;
      if (SWIGLU)
        Us[SWIGLU ? kk : 0][r] = (n0 + r < N && kin) ? to_f(B1[(size_t)(n0 + r) * K + gk]) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
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
      if (SWIGLU) {
        float u[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) u[j] = Us[SWIGLU ? kk : 0][tx + 16 * j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            acu[SWIGLU ? i : 0][j] = fmaf(a[i], u[j], acu[SWIGLU ? i : 0][j]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty + 16 * i;
    if (m >= rows) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx + 16 * j;
      if (n >= N) continue;
      const size_t o = (size_t)(row0 + m) * N + n;
      if (SWIGLU) {
        const float gv = acc[i][j];
        const float hv = gv / (1.f + expf(-gv)) * acu[SWIGLU ? i : 0][j];
        from_f(hv, (TIn*)(shared ? p.out_shared : p.out_routed) + o);
      } else {
        ((float*)(shared ? p.out_shared : p.out_routed))[o] = acc[i][j];
      }
    }
  }
}

template <typename TIn>
cudaError_t run(const moe_config_t& c, const ExpertArgs& a, cudaStream_t s) {
  const int E = c.n_experts, T = c.T, d = c.d_model, F = c.d_ff, Fs = c.d_ff_shared;
  const int has_shared = Fs > 0 && a.ws_gate != nullptr;
  const int max_rows = T;   // an expert holds each token at most once
  const int groups = E + (has_shared ? 1 : 0);
  SimtArgs p{};
  p.E = E;
  p.T = T;
  p.rows_cap = a.rows > 0 ? a.rows : T * c.top_k;
  p.offsets = a.offsets;
  p.has_shared = has_shared;
  // gate/up + SwiGLU: [rows, d] x [F, d]^T -> h [rows, F]
  p.a_routed = a.x_perm;
  p.a_shared = a.x;
  p.b0 = a.w_gate;
  p.b1 = a.w_up;
  p.bs0 = a.ws_gate;
  p.bs1 = a.ws_up;
  p.out_routed = a.h;
  p.out_shared = a.h_shared;
  p.K = d;
  p.N = F;
  p.K_s = d;
  p.N_s = Fs;
  const int nmax1 = F > Fs ? F : Fs;
  dim3 g1((nmax1 + 63) / 64, (max_rows + 63) / 64, groups);
  if (a.ev_up) {
    cudaError_t e = cudaEventRecord(a.ev_up, s);
    if (e != cudaSuccess) return e;
  }
  experts_simt_kernel<TIn, true><<<g1, 256, 0, s>>>(p);
  count_launch(a.launches);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  // down: h [rows, F] x [d, F]^T -> y [rows, d] fp32
  p.a_routed = a.h;
  p.a_shared = a.h_shared;
  p.b0 = a.w_down;
  p.b1 = nullptr;
  p.bs0 = a.ws_down;
  p.bs1 = nullptr;
  p.out_routed = a.y_perm;
  p.out_shared = a.y_shared;
  p.K = F;
  p.N = d;
  p.K_s = Fs;
  p.N_s = d;
  dim3 g2((d + 63) / 64, (max_rows + 63) / 64, groups);
  if (a.ev_down) {
    cudaError_t e = cudaEventRecord(a.ev_down, s);
    if (e != cudaSuccess) return e;
  }
  experts_simt_kernel<TIn, false><<<g2, 256, 0, s>>>(p);
  count_launch(a.launches);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_experts_simt(const moe_config_t& c, const ExpertArgs& a, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  if (c.act_dtype == MOE_BF16) return run<__nv_bfloat16>(c, a, s);
  return run<float>(c, a, s);
}

}  // namespace moe

// Self-test of the bounded-wait machinery that every tcgen05 kernel uses.
//
// One thread initialises an mbarrier that nothing will ever arrive on and
// waits for it through the same bounded wait (mbar_wait) the GEMMs use.  The
// wait must give up after `timeout_ns`, record the timeout in the workspace
// status word and let the kernel return, so the host can read the status
// with moe_get_error and keep using the CUDA context.
#include "tc_common.cuh"

namespace moe {
namespace {

__global__ void bounded_wait_selftest_kernel(int32_t* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = tc::smem_u32(&bar);
  if (threadIdx.x == 0) {
    tc::mbar_init(b, 1);
    tc::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // phase 0 never completes: no thread arrives on this barrier
    if (!tc::mbar_wait(b, 0, nullptr, timeout_ns)) record_error(status, kDevTimeout);
  }
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_selftest_bounded_wait(void* ws, size_t ws_bytes,
                                                  uint64_t timeout_ns, void* stream) {
  using namespace moe;
  if (!ws || ws_bytes < 256 || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return MOE_ERR_WORKSPACE;
  if (timeout_ns == 0 || timeout_ns > 1000000000ull) return MOE_ERR_INVALID_ARG;
  bounded_wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(static_cast<int32_t*>(ws),
                                                                  timeout_ns);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

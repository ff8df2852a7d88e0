// placeholder: replaced by the tcgen05 grouped GEMM
#include "internal.cuh"
namespace moe {
cudaError_t launch_experts_tc(const moe_config_t& c, const ExpertArgs& a, cudaStream_t s) {
  return launch_experts_simt(c, a, s);
}
}  // namespace moe

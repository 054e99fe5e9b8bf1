// Dispatch of the expert FFN kernels.
#include "experts.cuh"

namespace moe {

size_t tc_sched_bytes(const moe_dims& d);
cudaError_t launch_experts_tc(const ExpertsArgs& a, bool deterministic, cudaStream_t stream);

size_t experts_sched_bytes(const moe_dims& d) { return tc_sched_bytes(d); }

cudaError_t launch_experts_fast(const ExpertsArgs& a, uint32_t flags, cudaStream_t stream) {
  return launch_experts_tc(a, (flags & MOE_DETERMINISTIC) != 0, stream);
}

}  // namespace moe

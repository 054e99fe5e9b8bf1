// Dispatch of the expert FFN kernels.
#include "experts.cuh"

namespace moe {

size_t experts_sched_bytes(const moe_dims& d) { return 4096 + (size_t)(d.E + 1) * 64; }

cudaError_t launch_experts_fast(const ExpertsArgs& a, uint32_t flags, cudaStream_t stream) {
  return launch_experts_simple(a, (flags & MOE_DETERMINISTIC) != 0, stream);
}

}  // namespace moe

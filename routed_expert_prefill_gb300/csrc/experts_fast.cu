// Dispatch of the expert FFN kernels.
#include "experts.cuh"

namespace moe {

size_t tc_sched_bytes(const moe_dims& d);
cudaError_t launch_experts_tc(const ExpertsArgs& a, bool deterministic, cudaStream_t stream);

size_t packed_max_tiles(const moe_dims& d);

size_t experts_sched_bytes(const moe_dims& d) {
  // room for the larger (128-row) tile list of the packed-weight kernels
  const size_t mt = packed_max_tiles(d);
  const int fmax = (d.inter > d.shared_inter ? d.inter : d.shared_inter) / 128;
  const size_t packed = 64 + mt * 16 + mt * fmax * 4 + (size_t)d.t * 4 + 256;
  const size_t v2 = tc_sched_bytes(d);
  return packed > v2 ? packed : v2;
}

cudaError_t launch_experts_fast(const ExpertsArgs& a, uint32_t flags, cudaStream_t stream) {
  return launch_experts_tc(a, (flags & MOE_DETERMINISTIC) != 0, stream);
}

}  // namespace moe

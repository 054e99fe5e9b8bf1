// Streaming context of the routed records (internal): the residency plan
// and the state it keeps between chunks.
#pragma once
#include <cuda_runtime.h>

#include <vector>

#include "moe.h"

namespace moe {

// The plan of one chunk (moe_plan_residency); scratch vectors are reused
// across calls.  Returns MOE_OK or MOE_EINVAL (pool table inconsistent).
int plan_residency(const int32_t* counts, int E, const moe_stream_cfg& cfg, int64_t call, moe_residency_plan& plan);

}  // namespace moe

struct moe_streamer {
  int device;
  moe_dims dims;  // E, h, inter, bits fixed at creation (t and k vary per call)
  moe_stream_cfg cfg;
  size_t rec_bytes;  // one packed routed record at dims.bits (pool slots)
  int miss_bits;     // code width of the ring's records
  size_t miss_bytes; // one packed routed record at miss_bits (ring slots)
  int64_t call;      // call number of the last plan
  std::vector<int32_t> pool_expert;
  std::vector<int64_t> pool_last;
  // plan arrays
  std::vector<int32_t> counts, copy_expert, copy_slot, wait_for, plan_rec, plan_batch;
  int32_t* h_offsets = nullptr;  // pinned [E + 1]: the chunk's CSR offsets
  int32_t* h_maps = nullptr;     // pinned [2E + 1]: rec[E], batch_of[E + 1]
  int32_t* d_maps = nullptr;     // device copy of h_maps
  cudaStream_t copy = nullptr;   // fetch side
  cudaEvent_t fetched = nullptr;  // copy stream -> compute stream, per batch
  std::vector<cudaEvent_t> done;  // compute stream -> copy stream, batch b in done[b % lag]
  cudaEvent_t call_done = nullptr;  // end of the last call on its stream
  bool call_done_recorded = false;
  // the last call's first fetch batch when it held ring records only: the
  // next call fetches it again while it routes (expert, ring slot)
  std::vector<int32_t> spec_expert, spec_slot;
};

// Arguments and launchers of the expert-FFN kernels (internal).
#pragma once
#include "common.cuh"

namespace moe {

struct ExpertsArgs {
  const uint16_t* x;  // bf16 [t][h]
  int t, h, I, Is, E, k;
  int n_pairs;        // t*k: upper bound of the list length (the real one is offsets[E])
  const int32_t* offsets;
  const int32_t* rows;
  const float* weights;
  const int32_t* slot_of;
  const uint8_t* codes;  // [E][rec_bytes]
  const uint16_t* scales;
  const uint16_t* biases;
  size_t rec_bytes, rec_groups;
  const uint8_t* s_codes;  // shared record (may be null when Is == 0)
  const uint16_t* s_scales;
  const uint16_t* s_biases;
  const uint16_t* s_gate;  // bf16 [h] or null
  float* acc;              // fp32 [t][h]
  uint16_t* hg;            // bf16 [t*k][I]
  uint16_t* hgs;           // bf16 [t][Is]
  float* ybuf;             // fp32 [t*k][h] (deterministic only)
  unsigned char* sched;    // scheduler scratch
  DeviceStatus* status;
  uint16_t* out;           // bf16 [t][h]
};

cudaError_t launch_zero_f32(float* p, size_t n, cudaStream_t stream);
cudaError_t launch_finalize(const ExpertsArgs& a, bool deterministic, cudaStream_t stream);
cudaError_t launch_experts_simple(const ExpertsArgs& a, bool deterministic, cudaStream_t stream);

}  // namespace moe

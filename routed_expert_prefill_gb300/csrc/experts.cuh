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
  float* gvpart;           // small-t gate/up partial sums [4][t*k + t][2][max(I, Is)] (t <= 16)
  DeviceStatus* status;
  uint16_t* out;           // bf16 [t][h]
  int bits;                // code width of the records: 2, 3, 4 or 8 (packed kernels; the others take 4)
};

// Packed record layout (moe_pack_experts): 128-row x 64-K blocks of 4-bit
// codes (4096 bytes) + 128 bf16 scales + 128 bf16 biases; per record the
// gate/up part ([128-row tile][K chunk][gate block][up block]) then the down
// part ([128-row tile of h][K chunk of inter][block]).
constexpr int PACK_QB = 4096 + 256 + 256;
__host__ __device__ inline size_t packed_gu_bytes(int h, int I) { return (size_t)(I / 128) * (h / 64) * 2 * PACK_QB; }
__host__ __device__ inline size_t packed_rec_bytes(int h, int I) {
  return packed_gu_bytes(h, I) + (size_t)(h / 128) * (I / 64) * PACK_QB;
}

// One batch of a chunk whose routed records sit in record slots (streamed
// experts): only the experts e with batch_of[e] == batch (E = the shared
// expert) run, reading record rec_map[e] of n_rec.  The first batch zeroes
// the block accumulator and evaluates the shared gate; the last finalises.
struct PackedBatch {
  const int32_t* rec_map;
  int n_rec;
  const int32_t* batch_of;
  int batch;
  bool first, last;
};

cudaError_t launch_zero_f32(float* p, size_t n, cudaStream_t stream);
cudaError_t launch_finalize(const ExpertsArgs& a, bool deterministic, cudaStream_t stream);
cudaError_t launch_experts_simple(const ExpertsArgs& a, bool deterministic, cudaStream_t stream);

}  // namespace moe

// Types shared by the tensor-core expert kernels (internal).
#pragma once
#include <cuda.h>

#include "experts.cuh"

namespace moe {

struct SchedHdr {
  int n_tiles;
  int n_units_gu;
  int n_units_dn;
  int pad_rows;  // sum over tiles of the row count rounded up to 16
  int pad[12];
};

struct TcParams {
  int t, h, I, Is, E, k;
  int deterministic;
  const int32_t* offsets;
  const int32_t* rows;
  const float* weights;
  const uint16_t* scales;
  const uint16_t* biases;
  size_t rec_groups;
  const uint16_t* s_scales;
  const uint16_t* s_biases;
  const float* gate_vals;  // per-row shared-expert gate, or null
  float* acc;
  uint16_t* hg;
  uint16_t* hgs;
  float* ybuf;
  const SchedHdr* hdr;
  const int4* tiles;       // {expert (E = shared), start, rows, padded-row offset}
  const int* units_gu;     // (tile << 8) | feature tile
  DeviceStatus* status;
  int zero_acc;            // the gate/up kernel zeroes the fp32 block accumulator first
  // Expert subset (streamed records): when non-null, the schedule keeps only
  // the experts e (E = the shared expert) with batch_of[e] == batch.
  const int32_t* batch_of;
  int batch;
};


// Tile schedule: tiles of at most `tile_max` rows per expert (the shared
// expert: all t rows), largest first, with gate/up units and padded offsets.
cudaError_t launch_schedule(const TcParams& p, SchedHdr* hdr, int4* tiles, int* units_gu, int max_tiles,
                            int tile_max, cudaStream_t stream);
// 2D tiled tensor map over a row-major matrix: width (elements) x height
// (rows), row pitch in bytes, box {bw, bh}.
cudaError_t tmap_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t width, uint64_t height,
                    uint64_t stride_bytes, uint32_t bw, uint32_t bh, CUtensorMapSwizzle sw);
// Per-row shared-expert gate sigmoid(x_r . g) into out[t].
cudaError_t launch_shared_gate(const uint16_t* x, const uint16_t* g, int t, int h, float* out, cudaStream_t stream);

}  // namespace moe

// Tile schedule (internal), shared by the schedule kernel and the
// small-chunk preparation kernel: one block of 1024 threads.
#pragma once
#include "tc_common.cuh"

namespace moe {

// Tiles of at most `tile_max` rows per expert (the shared expert, index E:
// all t rows), largest first; gate/up units (tile << 8 | feature tile);
// padded-row offsets (rows rounded up to 16); the header.  Experts outside
// the batch filter (p.batch_of) get no tiles.
__device__ __forceinline__ void schedule_block(const TcParams& p, SchedHdr* hdr, int4* tiles, int* units_gu,
                                               int max_tiles, int tile_max) {
  __shared__ int bucket_cnt[16], bucket_base[16], bucket_fill[16];
  __shared__ int n_tiles_s;
  __shared__ int scan_carry;
  __shared__ int warp_sums[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nexp = p.E + (p.Is > 0 ? 1 : 0);
  if (tid < 16) {
    bucket_cnt[tid] = 0;
    bucket_fill[tid] = 0;
  }
  __syncthreads();
  // pass 1: count tiles per size bucket (bucket = ceil(size / 16) - 1)
  for (int e = tid; e < nexp; e += blockDim.x) {
    if (p.batch_of && p.batch_of[e] != p.batch) continue;
    int n;
    if (e < p.E) {
      n = p.offsets[e + 1] - p.offsets[e];
      if (n < 0 || p.offsets[e] < 0 || p.offsets[e + 1] > p.t * p.k) {
        raise_flag(p.status, FLAG_BAD_OFFSETS);
        n = 0;
      }
    } else {
      n = p.t;
    }
    if (n == 0) continue;
    const int nt = (n + tile_max - 1) / tile_max;
    const int sz = (n + nt - 1) / nt;
    for (int i = 0; i < nt; ++i) {
      const int rows = min(sz, n - i * sz);
      if (rows <= 0) break;
      atomicAdd(&bucket_cnt[(rows + 15) / 16 - 1], 1);
    }
  }
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int b = 15; b >= 0; --b) {  // largest tiles first
      bucket_base[b] = run;
      run += bucket_cnt[b];
    }
    n_tiles_s = min(run, max_tiles);
  }
  __syncthreads();
  // pass 2: place tiles
  for (int e = tid; e < nexp; e += blockDim.x) {
    if (p.batch_of && p.batch_of[e] != p.batch) continue;
    int n, start;
    if (e < p.E) {
      n = p.offsets[e + 1] - p.offsets[e];
      start = p.offsets[e];
      if (n < 0 || start < 0 || p.offsets[e + 1] > p.t * p.k) n = 0;
    } else {
      n = p.t;
      start = 0;
    }
    if (n == 0) continue;
    const int nt = (n + tile_max - 1) / tile_max;
    const int sz = (n + nt - 1) / nt;
    for (int i = 0; i < nt; ++i) {
      const int rows = min(sz, n - i * sz);
      if (rows <= 0) break;
      const int b = (rows + 15) / 16 - 1;
      const int pos = bucket_base[b] + atomicAdd(&bucket_fill[b], 1);
      if (pos < max_tiles) tiles[pos] = make_int4(e, start + i * sz, rows, 0);
    }
  }
  __syncthreads();
  // gate/up units: tile-major, feature tiles of 128 (I/128 routed, Is/128 shared)
  const int nt_all = n_tiles_s;
  if (tid == 0) scan_carry = 0;
  __syncthreads();
  for (int base = 0; base < nt_all; base += blockDim.x) {
    const int i = base + tid;
    int f = 0;
    if (i < nt_all) f = (tiles[i].x == p.E) ? p.Is / 128 : p.I / 128;
    int incl = f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int s = warp_sums[lane];
      int si = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xFFFFFFFFu, si, o);
        if (lane >= o) si += y;
      }
      warp_sums[lane] = si - s;
    }
    __syncthreads();
    const int ub = scan_carry + warp_sums[warp] + incl - f;
    for (int ft = 0; ft < f; ++ft) units_gu[ub + ft] = (i << 8) | ft;
    __syncthreads();
    if (tid == blockDim.x - 1) scan_carry = ub + f;
    __syncthreads();
  }
  const int n_units_gu = scan_carry;
  __syncthreads();
  // padded-row offset of every tile (rows rounded up to 16)
  if (tid == 0) scan_carry = 0;
  __syncthreads();
  for (int base = 0; base < nt_all; base += blockDim.x) {
    const int i = base + tid;
    const int f = (i < nt_all) ? (tiles[i].z + 15) & ~15 : 0;
    int incl = f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int s = warp_sums[lane];
      int si = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xFFFFFFFFu, si, o);
        if (lane >= o) si += y;
      }
      warp_sums[lane] = si - s;
    }
    __syncthreads();
    const int ub = scan_carry + warp_sums[warp] + incl - f;
    if (i < nt_all) tiles[i].w = ub;
    __syncthreads();
    if (tid == blockDim.x - 1) scan_carry = ub + f;
    __syncthreads();
  }
  if (tid == 0) {
    hdr->n_tiles = nt_all;
    hdr->n_units_gu = n_units_gu;
    hdr->n_units_dn = nt_all * (p.h / 128);
    hdr->pad_rows = scan_carry;
  }
}

}  // namespace moe

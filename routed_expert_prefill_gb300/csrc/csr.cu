// Expert grouping: the (row, slot) pairs of the router output as a CSR list
// in expert-ascending, row-ascending order (cherenkov qwen4_exp,
// prefill/experts.rs, prepare_expert_jobs: rows outer, slots inner, pushed
// onto per-expert lists that are then concatenated in expert order).
//
// The pairs p = r*k + j are already in that visiting order, so the list
// position of p is offsets[e] + (number of earlier pairs routed to e).  Three
// kernels compute it without atomics on the ordering:
//   1. csr_rank: each block of CSR_CHUNK consecutive pairs builds a bitmap
//      per expert in shared memory; a pair's rank inside its chunk is the
//      popcount of its expert's bits below it.  The block also writes its
//      per-expert counts.
//   2. csr_scan (one block): per expert, the exclusive prefix of the chunk
//      counts; then the exclusive prefix over experts gives offsets.
//   3. csr_scatter: position = offsets[e] + chunk prefix + rank.
// Up to CSR_SMALL_CHUNKS chunks run as one block that walks the chunks in
// order with running per-expert counts, scans them and scatters: one launch
// instead of three, the same positions.  Up to 256 pairs (decode steps) take
// a lighter one-block kernel (csr_tiny_kernel).
#include "common.cuh"

namespace moe {

namespace {

__global__ void __launch_bounds__(CSR_CHUNK)
csr_rank_kernel(const int32_t* __restrict__ idx, int n, int E, int32_t* __restrict__ rank,
                int32_t* __restrict__ counts, DeviceStatus* st) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint32_t bm[];  // [E][CSR_CHUNK / 32]
  constexpr int W = CSR_CHUNK / 32;
  const int tid = threadIdx.x;
  for (int i = tid; i < E * W; i += CSR_CHUNK) bm[i] = 0u;
  __syncthreads();
  const int p = blockIdx.x * CSR_CHUNK + tid;
  int e = -1;
  if (p < n) {
    e = idx[p];
    if (e < 0 || e >= E) {
      raise_flag(st, FLAG_BAD_EXPERT);
      e = -1;
    } else {
      atomicOr(&bm[e * W + (tid >> 5)], 1u << (tid & 31));
    }
  }
  __syncthreads();
  if (e >= 0) {
    const int wq = tid >> 5;
    int rk = __popc(bm[e * W + wq] & ((1u << (tid & 31)) - 1u));
    for (int q = 0; q < wq; ++q) rk += __popc(bm[e * W + q]);
    rank[p] = rk;
  }
  for (int ex = tid; ex < E; ex += CSR_CHUNK) {
    int c = 0;
#pragma unroll
    for (int q = 0; q < W; ++q) c += __popc(bm[ex * W + q]);
    counts[(size_t)blockIdx.x * E + ex] = c;
  }
}

__global__ void __launch_bounds__(1024)
csr_scan_kernel(const int32_t* __restrict__ counts, int nchunks, int E, int32_t* __restrict__ base,
                int32_t* __restrict__ offsets) {
  pdl_wait();
  pdl_trigger();
  __shared__ int32_t tot[1024];
  __shared__ int32_t warp_sums[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int run = 0;
  if (tid < E) {
    for (int c = 0; c < nchunks; ++c) {
      const int v = counts[(size_t)c * E + tid];
      base[(size_t)c * E + tid] = run;
      run += v;
    }
  }
  tot[tid] = (tid < E) ? run : 0;
  // Block-wide exclusive scan of tot.
  int v = tot[tid];
  int incl = v;
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
    warp_sums[lane] = si - s;  // exclusive prefix of warp sums
  }
  __syncthreads();
  const int excl = warp_sums[warp] + incl - v;
  if (tid < E) offsets[tid] = excl;
  if (tid == E - 1) offsets[E] = excl + v;
}

__global__ void csr_scatter_kernel(const int32_t* __restrict__ idx, const float* __restrict__ w, int n,
                                   int k, int E, const int32_t* __restrict__ rank,
                                   const int32_t* __restrict__ base, const int32_t* __restrict__ offsets,
                                   int32_t* __restrict__ rows, float* __restrict__ weights,
                                   int32_t* __restrict__ slot_of) {
  pdl_wait();
  pdl_trigger();
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= n) return;
  const int e = idx[p];
  if (e < 0 || e >= E) {
    slot_of[p] = -1;
    return;
  }
  const int c = p / CSR_CHUNK;
  const int pos = offsets[e] + base[(size_t)c * E + e] + rank[p];
  rows[pos] = p / k;
  weights[pos] = w[p];
  slot_of[p] = pos;
}


constexpr int CSR_SMALL_CHUNKS = 2;

// Exclusive scan over v[0..1023] held one per thread (1024 threads); returns
// this thread's exclusive prefix and, in *total, the sum.
__device__ __forceinline__ int block_excl_scan_1024(int v, int* warp_sums, int* total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int s = warp_sums[lane];
    int si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xFFFFFFFFu, si, o);
      if (lane >= o) si += y;
    }
    warp_sums[lane] = si - s;
    if (lane == 31) warp_sums[32] = si;
  }
  __syncthreads();
  *total = warp_sums[32];
  return warp_sums[warp] + incl - v;
}

// Up to CSR_TINY pairs (decode steps): one 256-thread block.  Per-expert
// counts by shared atomics, one exclusive scan over the experts (four per
// thread), and each pair's rank inside its expert by counting the earlier
// pairs of the same expert: the same stable order as the chunked kernels.
constexpr int CSR_TINY = 256;

__global__ void __launch_bounds__(CSR_TINY, 1)
csr_tiny_kernel(const int32_t* __restrict__ idx, const float* __restrict__ w, int n, int k, int E,
                int32_t* __restrict__ offsets, int32_t* __restrict__ rows, float* __restrict__ weights,
                int32_t* __restrict__ slot_of, DeviceStatus* st) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int start[];  // [E]: the expert's count, then its list start
  __shared__ int es[CSR_TINY];
  __shared__ int warp_sums[CSR_TINY / 32 + 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < E; i += CSR_TINY) start[i] = 0;
  int e = -1;
  if (tid < n) {
    e = idx[tid];
    if (e < 0 || e >= E) {
      raise_flag(st, FLAG_BAD_EXPERT);
      e = -1;
    }
  }
  es[tid] = e;
  __syncthreads();
  if (e >= 0) atomicAdd(&start[e], 1);
  __syncthreads();
  // exclusive scan over the experts; thread tid owns experts 4 tid .. 4 tid + 3
  int c[4], sum = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int ex = 4 * tid + j;
    c[j] = ex < E ? start[ex] : 0;
    sum += c[j];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int sv = lane < CSR_TINY / 32 ? warp_sums[lane] : 0;
    int si = sv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, si, o);
      if (lane >= o) si += y;
    }
    if (lane < CSR_TINY / 32) warp_sums[lane] = si - sv;
    if (lane == CSR_TINY / 32 - 1) warp_sums[CSR_TINY / 32] = si;
  }
  __syncthreads();
  int run = warp_sums[warp] + incl - sum;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int ex = 4 * tid + j;
    if (ex < E) {
      start[ex] = run;
      offsets[ex] = run;
    }
    run += c[j];
  }
  if (tid == 0) offsets[E] = warp_sums[CSR_TINY / 32];
  __syncthreads();
  if (tid < n) {
    if (e < 0) {
      slot_of[tid] = -1;
    } else {
      int r = 0;
      for (int q = 0; q < tid; ++q) r += es[q] == e;
      const int pos = start[e] + r;
      rows[pos] = tid / k;
      weights[pos] = w[tid];
      slot_of[tid] = pos;
    }
  }
}

__global__ void __launch_bounds__(CSR_CHUNK, 1)
csr_small_kernel(const int32_t* __restrict__ idx, const float* __restrict__ w, int n, int k, int E,
                 int32_t* __restrict__ offsets, int32_t* __restrict__ rows, float* __restrict__ weights,
                 int32_t* __restrict__ slot_of, DeviceStatus* st) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint32_t sm[];
  constexpr int W = CSR_CHUNK / 32;
  uint32_t* bm = sm;                                      // [E][W] chunk bitmap
  int* run = reinterpret_cast<int*>(sm + E * W);          // [E] pairs seen per expert
  uint16_t* pre = reinterpret_cast<uint16_t*>(run + E);   // [E][W] bits of the expert in earlier words
  __shared__ int warp_sums[33];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nch = (n + CSR_CHUNK - 1) / CSR_CHUNK;
  for (int i = tid; i < E; i += CSR_CHUNK) run[i] = 0;
  int ee[CSR_SMALL_CHUNKS], pe[CSR_SMALL_CHUNKS];
#pragma unroll
  for (int c = 0; c < CSR_SMALL_CHUNKS; ++c) {
    ee[c] = -1;
    pe[c] = 0;
    if (c < nch) {
      for (int i = tid; i < E * W; i += CSR_CHUNK) bm[i] = 0u;
      __syncthreads();
      const int p = c * CSR_CHUNK + tid;
      int e = -1;
      if (p < n) {
        e = idx[p];
        if (e < 0 || e >= E) {
          raise_flag(st, FLAG_BAD_EXPERT);
          e = -1;
        } else {
          atomicOr(&bm[e * W + (tid >> 5)], 1u << (tid & 31));
        }
      }
      __syncthreads();
      // per expert (one warp each): exclusive prefix of its bit counts over the W words
      for (int ex = warp; ex < E; ex += CSR_CHUNK / 32) {
        const int cnt = __popc(bm[ex * W + lane]);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += y;
        }
        pre[ex * W + lane] = (uint16_t)(incl - cnt);
      }
      __syncthreads();
      if (e >= 0) pe[c] = run[e] + pre[e * W + warp] + __popc(bm[e * W + warp] & ((1u << lane) - 1u));
      ee[c] = e;
      __syncthreads();
      for (int ex = tid; ex < E; ex += CSR_CHUNK) run[ex] += pre[ex * W + W - 1] + __popc(bm[ex * W + W - 1]);
      __syncthreads();
    }
  }
  // offsets: exclusive prefix of the per-expert totals (E <= 1024 = one per thread)
  int total;
  const int excl = block_excl_scan_1024(tid < E ? run[tid] : 0, warp_sums, &total);
  __syncthreads();
  if (tid < E) {
    offsets[tid] = excl;
    run[tid] = excl;  // reused as the expert's list start
  }
  if (tid == 0) offsets[E] = total;
  __syncthreads();
#pragma unroll
  for (int c = 0; c < CSR_SMALL_CHUNKS; ++c) {
    const int p = c * CSR_CHUNK + tid;
    if (c < nch && p < n) {
      if (ee[c] < 0) {
        slot_of[p] = -1;
      } else {
        const int pos = run[ee[c]] + pe[c];
        rows[pos] = p / k;
        weights[pos] = w[p];
        slot_of[p] = pos;
      }
    }
  }
}

}  // namespace

cudaError_t launch_build_csr(const int32_t* idx, const float* w, int t, int k, int E,
                             const moe_csr& csr, unsigned char* ws, const WsLayout& L,
                             cudaStream_t stream) {
  const int n = t * k;
  const int nchunks = (n + CSR_CHUNK - 1) / CSR_CHUNK;
  int32_t* rank = reinterpret_cast<int32_t*>(ws + L.csr_rank);
  int32_t* counts = reinterpret_cast<int32_t*>(ws + L.csr_counts);
  int32_t* base = reinterpret_cast<int32_t*>(ws + L.csr_base);
  DeviceStatus* st = reinterpret_cast<DeviceStatus*>(ws + L.status);
  if (n <= CSR_TINY && E <= 4 * CSR_TINY) {
    MOE_LAUNCH("csr_tiny", stream,
               launch_k(csr_tiny_kernel, 1, CSR_TINY, (size_t)E * 4, stream, idx, w, n, k, E, csr.offsets, csr.rows,
                        csr.weights, csr.slot_of, st));
    return cudaGetLastError();
  }
  if (nchunks <= CSR_SMALL_CHUNKS) {
    const size_t smem = (size_t)E * (CSR_CHUNK / 32) * 6 + (size_t)E * 4;
    cudaError_t err =
        set_smem_limit_once(csr_small_kernel, (int)smem);
    if (err != cudaSuccess) return err;
    MOE_LAUNCH("csr_small", stream,
               launch_k(csr_small_kernel, 1, CSR_CHUNK, smem, stream, idx, w, n, k, E, csr.offsets, csr.rows, csr.weights,
                                                                csr.slot_of, st));
    return cudaGetLastError();
  }
  const size_t smem = (size_t)E * (CSR_CHUNK / 32) * 4;
  cudaError_t err = set_smem_limit_once(csr_rank_kernel, (int)smem);
  if (err != cudaSuccess) return err;
  MOE_LAUNCH("csr_rank", stream,
             launch_k(csr_rank_kernel, nchunks, CSR_CHUNK, smem, stream, idx, n, E, rank, counts, st));
  MOE_LAUNCH("csr_scan", stream, launch_k(csr_scan_kernel, 1, 1024, 0, stream, counts, nchunks, E, base, csr.offsets));
  MOE_LAUNCH("csr_scatter", stream,
             launch_k(csr_scatter_kernel, (n + 255) / 256, 256, 0, stream, idx, w, n, k, E, rank, base, csr.offsets,
                                                                    csr.rows, csr.weights, csr.slot_of));
  return cudaGetLastError();
}

}  // namespace moe

// ----------------------------------------------------------------------------
// moe_build_csr_noalloc: the same grouping for callers that cannot allocate
// device memory (a caller already inside a memory pool it does not own, an
// embedding that forbids cudaMalloc on its hot path, ...).  Its scratch is a
// fixed array in this library's device image, so each GPU that loads the
// library holds it (NOALLOC_SCRATCH_BYTES) until the process exits.
// ----------------------------------------------------------------------------
namespace moe {

namespace {

constexpr size_t NOALLOC_RANK_OFF = 256;  // after the status flags
constexpr size_t NOALLOC_COUNTS_OFF = NOALLOC_RANK_OFF + (size_t)MOE_NOALLOC_MAX_PAIRS * 4;
constexpr size_t NOALLOC_BASE_OFF = NOALLOC_COUNTS_OFF + (size_t)MOE_NOALLOC_MAX_PAIRS * 4;
constexpr size_t NOALLOC_SCRATCH_BYTES = NOALLOC_BASE_OFF + (size_t)MOE_NOALLOC_MAX_PAIRS * 4;

// Status flags, per-pair ranks, per-chunk counts and prefixes.  The count
// table holds E * ceil(t*k / CSR_CHUNK) entries, which is at most
// 1024 * MOE_NOALLOC_MAX_PAIRS / 1024 = MOE_NOALLOC_MAX_PAIRS.
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

}  // namespace

}  // namespace moe

extern "C" int moe_noalloc_read_status(void* stream) {
  using namespace moe;
  void* p = nullptr;
  cudaError_t err = cudaGetSymbolAddress(&p, moe::g_noalloc_scratch);
  if (err != cudaSuccess) return set_error(MOE_ECUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(err));
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t flags = 0;
  if ((err = cudaMemcpyAsync(&flags, p, sizeof(flags), cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
      (err = cudaStreamSynchronize(s)) != cudaSuccess ||
      (err = cudaMemsetAsync(p, 0, sizeof(DeviceStatus), s)) != cudaSuccess ||
      (err = cudaStreamSynchronize(s)) != cudaSuccess)
    return set_error(MOE_ECUDA, "moe_noalloc_read_status: %s", cudaGetErrorString(err));
  if (flags & (FLAG_BAD_EXPERT | FLAG_BAD_ROW | FLAG_BAD_OFFSETS))
    return set_error(MOE_EDEVICE, "moe_build_csr_noalloc: expert id out of range (flags 0x%x)", flags);
  return MOE_OK;
}

extern "C" int moe_build_csr_noalloc(const int32_t* idx, const float* w, const moe_dims* dims, const moe_csr* csr,
                                     void* stream) {
  using namespace moe;
  if (!dims) return set_error(MOE_EINVAL, "dims is NULL");
  if (dims->t < 1 || dims->k < 1 || dims->k > 16 || dims->E < 1 || dims->E > 1024 || dims->k > dims->E)
    return set_error(MOE_ESHAPE, "t=%d, k=%d, E=%d outside 1 <= t, 1 <= k <= min(E, 16), E <= 1024", dims->t,
                     dims->k, dims->E);
  if ((long long)dims->t * dims->k > MOE_NOALLOC_MAX_PAIRS)
    return set_error(MOE_ESHAPE, "t*k = %lld exceeds the %d pairs moe_build_csr_noalloc's fixed scratch holds",
                     (long long)dims->t * dims->k, MOE_NOALLOC_MAX_PAIRS);
  if (!idx || !w || !csr || !csr->offsets || !csr->rows || !csr->weights || !csr->slot_of)
    return set_error(MOE_EINVAL, "a pointer argument is NULL");
  const void* ptrs[] = {idx, w, csr->offsets, csr->rows, csr->weights, csr->slot_of};
  for (const void* p : ptrs)
    if ((uintptr_t)p % 4) return set_error(MOE_EINVAL, "a pointer argument is not 4-byte aligned");

  // The device address of the array, looked up on every call: after a
  // device reset or a re-created primary context the module is loaded anew
  // and a cached address would be stale (the lookup is cheap once loaded).
  unsigned char* scratch;
  {
    void* p = nullptr;
    cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess) return set_error(MOE_ECUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(err));
    scratch = static_cast<unsigned char*>(p);
  }
  cudaError_t err;
  cudaStream_t s = (cudaStream_t)stream;
  // The status flags are OR-ed into and kept until moe_noalloc_read_status
  // clears them; everything else is written before it is read.
  WsLayout L{};
  L.status = 0;
  L.csr_rank = NOALLOC_RANK_OFF;
  L.csr_counts = NOALLOC_COUNTS_OFF;
  L.csr_base = NOALLOC_BASE_OFF;
  err = launch_build_csr(idx, w, dims->t, dims->k, dims->E, *csr, scratch, L, s);
  if (err != cudaSuccess) return set_error(MOE_ECUDA, "moe_build_csr_noalloc launch: %s", cudaGetErrorString(err));
  return MOE_OK;
}

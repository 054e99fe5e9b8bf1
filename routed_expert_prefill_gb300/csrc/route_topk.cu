// Router: logits, top-k and weights for every row of a chunk
// (cherenkov qwen4_exp, prefill.rs, pf_layer -> router_b).
//
// One CTA owns RT_ROWS rows.  Its 8 warps each compute an RT_ROWS x RT_EXW
// tile of logits per pass over the experts.  Lane l of a warp owns the K
// indices 256*m + 8*l + c and accumulates, for every (row, expert) of the
// tile, the exact bf16*bf16 products in fp32 with m ascending and c
// ascending; the 32 lane sums are then combined with the xor butterfly
// (offsets 16, 8, 4, 2, 1).  This is the summation order the header
// specifies, so logits are reproducible bit for bit.  x rows stay in shared
// memory; router weight chunks [64 experts][256 K] are double-buffered with
// cp.async.  After all passes, warp w selects the top-k of row w.
#include "route_common.cuh"

namespace moe {

namespace {

constexpr int RT_ROWS = 8;
constexpr int RT_EXW = 8;
constexpr int RT_WARPS = 8;
constexpr int RT_THREADS = RT_WARPS * 32;
constexpr int RT_PASS = RT_EXW * RT_WARPS;  // experts per pass
constexpr int KSPAN = 256;                  // K indices per step: 32 lanes x 8

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  int n = valid ? 16 : 0;  // src-size 0 -> zero fill
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__global__ void __launch_bounds__(RT_THREADS, 1)
route_topk_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr,
                  const float* __restrict__ rbias, int t, int h, int E, int k,
                  int32_t* __restrict__ idx, float* __restrict__ wout,
                  float* __restrict__ logits) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char smem[];
  const int hp = (h + KSPAN - 1) / KSPAN * KSPAN;
  const int nm = hp / KSPAN;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);                 // [RT_ROWS][hp]
  uint16_t* wsm = xs + RT_ROWS * hp;                                 // [2][RT_PASS][KSPAN]
  float* lg = reinterpret_cast<float*>(wsm + 2 * RT_PASS * KSPAN);  // [RT_ROWS][E]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row0 = blockIdx.x * RT_ROWS;
  const int vpr = hp / 8;  // 16-byte vectors per staged row

  for (int v = tid; v < RT_ROWS * vpr; v += RT_THREADS) {
    int r = v / vpr, c = v - r * vpr;
    bool ok = (row0 + r < t) && (c * 8 < h);
    cp_async16(xs + (size_t)v * 8, ok ? (const void*)(x + (size_t)(row0 + r) * h + c * 8) : (const void*)x, ok);
  }
  cp_async_commit();

  auto stage_w = [&](int e0, int m, int buf) {
    uint16_t* dst = wsm + buf * RT_PASS * KSPAN;
    for (int v = tid; v < RT_PASS * (KSPAN / 8); v += RT_THREADS) {
      int e = v / (KSPAN / 8), c = v - e * (KSPAN / 8);
      int i = m * KSPAN + c * 8;
      bool ok = (e0 + e < E) && (i < h);
      cp_async16(dst + (size_t)v * 8, ok ? (const void*)(wr + (size_t)(e0 + e) * h + i) : (const void*)wr, ok);
    }
    cp_async_commit();
  };

  const int npass = (E + RT_PASS - 1) / RT_PASS;
  const int nsteps = npass * nm;
  stage_w(0, 0, 0);

  float P[RT_ROWS][RT_EXW];
  for (int s = 0; s < nsteps; ++s) {
    const int pass = s / nm, m = s - pass * nm;
    if (m == 0) {
#pragma unroll
      for (int r = 0; r < RT_ROWS; ++r)
#pragma unroll
        for (int j = 0; j < RT_EXW; ++j) P[r][j] = 0.f;
    }
    if (s + 1 < nsteps) {
      const int s1 = s + 1, p1 = s1 / nm;
      stage_w(p1 * RT_PASS, s1 - p1 * nm, s1 & 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    const uint4* xv4 = reinterpret_cast<const uint4*>(xs);
    const uint4* wv4 = reinterpret_cast<const uint4*>(wsm + (s & 1) * RT_PASS * KSPAN);
    uint4 xv[RT_ROWS], wv[RT_EXW];
#pragma unroll
    for (int r = 0; r < RT_ROWS; ++r) xv[r] = xv4[r * vpr + m * 32 + lane];
#pragma unroll
    for (int j = 0; j < RT_EXW; ++j) wv[j] = wv4[(warp * RT_EXW + j) * 32 + lane];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      float xf[RT_ROWS], wf[RT_EXW];
#pragma unroll
      for (int r = 0; r < RT_ROWS; ++r) {
        uint32_t word = (&xv[r].x)[c >> 1];
        xf[r] = (c & 1) ? bf16hi(word) : bf16lo(word);
      }
#pragma unroll
      for (int j = 0; j < RT_EXW; ++j) {
        uint32_t word = (&wv[j].x)[c >> 1];
        wf[j] = (c & 1) ? bf16hi(word) : bf16lo(word);
      }
      // The product of two bf16 values is exact in fp32, so the fma rounds
      // exactly once, like "sum + product".
#pragma unroll
      for (int r = 0; r < RT_ROWS; ++r)
#pragma unroll
        for (int j = 0; j < RT_EXW; ++j) P[r][j] = fmaf(xf[r], wf[j], P[r][j]);
    }

    if (m == nm - 1) {
      const int e0 = pass * RT_PASS + warp * RT_EXW;
#pragma unroll
      for (int r = 0; r < RT_ROWS; ++r)
#pragma unroll
        for (int j = 0; j < RT_EXW; ++j) {
          float v = P[r][j];
          v = v + __shfl_xor_sync(0xFFFFFFFFu, v, 16);
          v = v + __shfl_xor_sync(0xFFFFFFFFu, v, 8);
          v = v + __shfl_xor_sync(0xFFFFFFFFu, v, 4);
          v = v + __shfl_xor_sync(0xFFFFFFFFu, v, 2);
          v = v + __shfl_xor_sync(0xFFFFFFFFu, v, 1);
          const int e = e0 + j;
          if (lane == 0 && e < E) lg[r * E + e] = rbias ? v + rbias[e] : v;
        }
    }
    __syncthreads();  // buffer (s & 1) is refilled at step s + 2
  }

  if (logits) {
    for (int v = tid; v < RT_ROWS * E; v += RT_THREADS) {
      int r = v / E, e = v - r * E;
      if (row0 + r < t) logits[(size_t)(row0 + r) * E + e] = lg[v];
    }
  }

  // Top-k of row `warp`: keys order by (logit, -expert id).
  const int r = warp;
  if (row0 + r >= t) return;
  const float* lr = lg + r * E;
  uint64_t key[32];
#pragma unroll
  for (int q = 0; q < 32; ++q) {
    int e = lane + 32 * q;
    key[q] = (e < E) ? topk_key(lr[e], e) : 0ull;
  }
  warp_topk_softmax<32>(key, k, lane, idx + (size_t)(row0 + r) * k, wout + (size_t)(row0 + r) * k);
}

}  // namespace

size_t route_smem_bytes(int h, int E) {
  const int hp = (h + KSPAN - 1) / KSPAN * KSPAN;
  return (size_t)RT_ROWS * hp * 2 + (size_t)2 * RT_PASS * KSPAN * 2 + (size_t)RT_ROWS * E * 4;
}

cudaError_t launch_route_topk(const uint16_t* x, const uint16_t* wr, const float* rbias, int t,
                              int h, int E, int k, int32_t* idx, float* w, float* logits,
                              cudaStream_t stream) {
  const size_t smem = route_smem_bytes(h, E);
  cudaError_t err = set_smem_limit_once(route_topk_kernel, (int)smem);
  if (err != cudaSuccess) return err;
  dim3 grid((t + RT_ROWS - 1) / RT_ROWS);
  MOE_LAUNCH("route_topk", stream,
             launch_k(route_topk_kernel, grid, RT_THREADS, smem, stream, x, wr, rbias, t, h, E, k, idx, w, logits));
  return cudaGetLastError();
}

}  // namespace moe

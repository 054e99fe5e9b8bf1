// Plain CUDA-core expert FFNs: one block per CSR list position (or per row
// for the shared expert), warps over output features, lanes over K.  Slow,
// but with the same rounding points as the tensor-core kernels (bf16 fma
// dequantisation, fp32 accumulation, bf16 silu(gate)*up, fp32 block sum), so
// it serves as an independent GPU cross-check of the fast path.
//
// The steps follow cherenkov qwen4_exp, prefill/experts.rs, pf_experts:
// shared expert into the block output, then per list position: gather the
// row, gate and up quantised matmuls, silu_mul, down quantised matmul, and
// scatter_add_rows with the routing weight.
#include "common.cuh"
#include "experts.cuh"

namespace moe {

namespace {

constexpr int SB = 256;  // threads per block

__device__ __forceinline__ int expert_of(const int32_t* offsets, int E, int p) {
  // largest e with offsets[e] <= p (offsets nondecreasing, offsets[0] = 0)
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (offsets[mid] <= p) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + expf(-g)) * u; }

// Dot product of a staged fp32 vector with one quantised row (K values).
__device__ __forceinline__ float qrow_dot(const float* xs, const uint8_t* codes, const uint16_t* sc,
                                          const uint16_t* bi, int K, int lane) {
  float acc = 0.f;
  for (int kk = lane * 8; kk < K; kk += 256) {
    uint32_t word = *reinterpret_cast<const uint32_t*>(codes + kk / 2);
    const int g = kk / 64;
    __nv_bfloat16 s = h2bf(sc[g]), b = h2bf(bi[g]);
    uint32_t wq[4];
    dequant8(word, __halves2bfloat162(s, s), __halves2bfloat162(b, b), wq);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      float wv = (c & 1) ? bf16hi(wq[c >> 1]) : bf16lo(wq[c >> 1]);
      acc = fmaf(xs[kk + c], wv, acc);
    }
  }
  return acc;
}

__global__ void __launch_bounds__(SB)
gateup_simple_kernel(ExpertsArgs a, int shared) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float xs[];
  const int p = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = a.h;
  const int I = shared ? a.Is : a.I;
  int row;
  const uint8_t* codes;
  const uint16_t *sc, *bi;
  if (shared) {
    row = p;
    codes = a.s_codes;
    sc = a.s_scales;
    bi = a.s_biases;
  } else {
    if (p >= a.offsets[a.E]) return;  // list shorter than t*k (dropped pairs)
    const int e = expert_of(a.offsets, a.E, p);
    row = a.rows[p];
    codes = a.codes + (size_t)e * a.rec_bytes;
    sc = a.scales + (size_t)e * a.rec_groups;
    bi = a.biases + (size_t)e * a.rec_groups;
  }
  uint16_t* hg = shared ? a.hgs + (size_t)p * I : a.hg + (size_t)p * I;
  if (row < 0 || row >= a.t) {
    if (tid == 0) raise_flag(a.status, FLAG_BAD_ROW);
    for (int o = tid; o < I; o += SB) hg[o] = 0;
    return;
  }
  for (int i = tid; i < h; i += SB) xs[i] = bf16f(a.x[(size_t)row * h + i]);
  __syncthreads();
  const size_t mat_bytes = (size_t)I * h / 2, mat_groups = (size_t)I * h / 64;
  for (int o = warp; o < I; o += SB / 32) {
    float g = qrow_dot(xs, codes + (size_t)o * h / 2, sc + (size_t)o * (h / 64), bi + (size_t)o * (h / 64), h, lane);
    float u = qrow_dot(xs, codes + mat_bytes + (size_t)o * h / 2, sc + mat_groups + (size_t)o * (h / 64),
                       bi + mat_groups + (size_t)o * (h / 64), h, lane);
    g = warp_sum(g);
    u = warp_sum(u);
    if (lane == 0) hg[o] = f2bf(silu_mul(g, u));
  }
}

// mode 0: routed, fp32 atomics into acc; mode 1: routed, unweighted y into ybuf
// mode 2: shared, store g_r * y into acc.
__global__ void __launch_bounds__(SB)
down_simple_kernel(ExpertsArgs a, int mode) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float hs[];
  __shared__ float gate_r;
  const int p = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = a.h;
  const bool shared = (mode == 2);
  const int I = shared ? a.Is : a.I;
  int row;
  float wgt = 1.f;
  const uint8_t* codes;
  const uint16_t *sc, *bi;
  if (shared) {
    row = p;
    codes = a.s_codes + (size_t)2 * I * h / 2;
    sc = a.s_scales + (size_t)2 * I * h / 64;
    bi = a.s_biases + (size_t)2 * I * h / 64;
  } else {
    if (p >= a.offsets[a.E]) return;
    const int e = expert_of(a.offsets, a.E, p);
    row = a.rows[p];
    wgt = a.weights[p];
    codes = a.codes + (size_t)e * a.rec_bytes + (size_t)2 * I * h / 2;
    sc = a.scales + (size_t)e * a.rec_groups + (size_t)2 * I * h / 64;
    bi = a.biases + (size_t)e * a.rec_groups + (size_t)2 * I * h / 64;
  }
  if (row < 0 || row >= a.t) {
    if (tid == 0) raise_flag(a.status, FLAG_BAD_ROW);
    if (mode == 1)
      for (int f = tid; f < h; f += SB) a.ybuf[(size_t)p * h + f] = 0.f;
    return;
  }
  const uint16_t* hrow = shared ? a.hgs + (size_t)p * I : a.hg + (size_t)p * I;
  for (int i = tid; i < I; i += SB) hs[i] = bf16f(hrow[i]);
  if (shared && warp == 0) {
    float gr = 1.f;
    if (a.s_gate) {
      float d = 0.f;
      for (int i = lane; i < h; i += 32) d = fmaf(bf16f(a.x[(size_t)row * h + i]), bf16f(a.s_gate[i]), d);
      d = warp_sum(d);
      gr = 1.f / (1.f + expf(-d));
    }
    if (lane == 0) gate_r = gr;
  }
  __syncthreads();
  for (int f = warp; f < h; f += SB / 32) {
    float y = qrow_dot(hs, codes + (size_t)f * I / 2, sc + (size_t)f * (I / 64), bi + (size_t)f * (I / 64), I, lane);
    y = warp_sum(y);
    if (lane == 0) {
      if (mode == 0) atomicAdd(&a.acc[(size_t)row * h + f], wgt * y);
      else if (mode == 1) a.ybuf[(size_t)p * h + f] = y;
      else a.acc[(size_t)row * h + f] = gate_r * y;
    }
  }
}

}  // namespace

cudaError_t launch_experts_simple(const ExpertsArgs& a, bool deterministic, cudaStream_t stream) {
  cudaError_t err;
  const int n = a.n_pairs;
  const int smax = (a.h > a.I ? a.h : a.I) * 4;
  if ((err = set_smem_limit_once(gateup_simple_kernel, smax)) != cudaSuccess)
    return err;
  if ((err = set_smem_limit_once(down_simple_kernel, (a.I > a.Is ? a.I : a.Is) * 4)) != cudaSuccess)
    return err;
  if (a.Is > 0) {
    MOE_LAUNCH("gateup_simple", stream, launch_k(gateup_simple_kernel, a.t, SB, a.h * 4, stream, a, 1));
    MOE_LAUNCH("down_simple", stream, launch_k(down_simple_kernel, a.t, SB, a.Is * 4, stream, a, 2));
  } else {
    err = launch_zero_f32(a.acc, (size_t)a.t * a.h, stream);
    if (err != cudaSuccess) return err;
  }
  if (n > 0) {
    MOE_LAUNCH("gateup_simple", stream, launch_k(gateup_simple_kernel, n, SB, a.h * 4, stream, a, 0));
    MOE_LAUNCH("down_simple", stream, launch_k(down_simple_kernel, n, SB, a.I * 4, stream, a, deterministic ? 1 : 0));
  }
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  return launch_finalize(a, deterministic, stream);
}

}  // namespace moe

// Block-output initialisation and the final fp32 -> bf16 pass.
#include "experts.cuh"

namespace moe {

namespace {

__global__ void zero_f32_kernel(float4* __restrict__ p, size_t n4) {
  pdl_wait();
  pdl_trigger();
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x)
    p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// out[r] = bf16(acc[r]) (atomic mode), or, deterministic mode,
// out[r] = bf16(acc[r] + sum over the row's list positions in ascending order
// (= expert-ascending) of weight * y), acc holding the shared term.
__global__ void __launch_bounds__(256)
finalize_kernel(ExpertsArgs a, int deterministic) {
  pdl_wait();
  pdl_trigger();
  __shared__ int pos[16];
  __shared__ int npos;
  const int r = blockIdx.x;
  const int h = a.h;
  if (deterministic && threadIdx.x == 0) {
    int m = 0;
    for (int j = 0; j < a.k; ++j) {
      const int p = a.slot_of[(size_t)r * a.k + j];
      if (p < 0) continue;
      int i = m++;
      while (i > 0 && pos[i - 1] > p) { pos[i] = pos[i - 1]; --i; }
      pos[i] = p;
    }
    npos = m;
  }
  __syncthreads();
  for (int f4 = threadIdx.x; f4 < h / 4; f4 += blockDim.x) {
    float4 v = reinterpret_cast<const float4*>(a.acc + (size_t)r * h)[f4];
    if (deterministic) {
      for (int j = 0; j < npos; ++j) {
        const float w = a.weights[pos[j]];
        const float4 y = reinterpret_cast<const float4*>(a.ybuf + (size_t)pos[j] * h)[f4];
        v.x = fmaf(w, y.x, v.x);
        v.y = fmaf(w, y.y, v.y);
        v.z = fmaf(w, y.z, v.z);
        v.w = fmaf(w, y.w, v.w);
      }
    }
    uint2 o;
    o.x = pack_bf16x2(v.x, v.y);
    o.y = pack_bf16x2(v.z, v.w);
    reinterpret_cast<uint2*>(a.out + (size_t)r * h)[f4] = o;
  }
}

}  // namespace

cudaError_t launch_zero_f32(float* p, size_t n, cudaStream_t stream) {
  const size_t n4 = n / 4;  // callers pass multiples of 4
  int blocks = (int)((n4 + 255) / 256);
  if (blocks > 152 * 8) blocks = 152 * 8;
  if (blocks < 1) blocks = 1;
  MOE_LAUNCH("zero_acc", stream, launch_k(zero_f32_kernel, blocks, 256, 0, stream, reinterpret_cast<float4*>(p), n4));
  return cudaGetLastError();
}

cudaError_t launch_finalize(const ExpertsArgs& a, bool deterministic, cudaStream_t stream) {
  MOE_LAUNCH("finalize", stream, launch_k(finalize_kernel, a.t, 256, 0, stream, a, deterministic ? 1 : 0));
  return cudaGetLastError();
}

}  // namespace moe

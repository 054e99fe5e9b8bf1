// Router pieces shared by the exact single-pass kernel and the
// tensor-core scoring + exact refinement kernels, so that both select and
// weight the experts with the same instructions (prefill.rs, pf_layer ->
// router_b: top-k of the logits, then a softmax over the selected ones).
#pragma once
#include "common.cuh"

namespace moe {

// Total order on floats as unsigned keys (larger float -> larger key).
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

// 64-bit selection key: logit first, then the lower expert id.
__device__ __forceinline__ uint64_t topk_key(float logit, int e) {
  return ((uint64_t)float_key(logit) << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)e);
}

// Warp-wide top-k over the keys key[q] (expert lane + 32 q; 0 = absent):
// lane j keeps the j-th selected expert; the softmax over the selected
// logits sums exp(l_j - l_0) for j = 0..k-1 in that order.  Lanes 0..k-1
// write idx and w.
template <int NQ>
__device__ __forceinline__ void warp_topk_softmax(uint64_t (&key)[NQ], int k, int lane, int32_t* idx_row,
                                                  float* w_row) {
  int my_e = 0;
  float my_l = 0.f;
  for (int j = 0; j < k; ++j) {
    uint64_t best = 0;
#pragma unroll
    for (int q = 0; q < NQ; ++q) best = key[q] > best ? key[q] : best;
    // the warp's largest key, in two 32-bit reductions: the logit part,
    // then the expert part among the lanes that hold that logit
    const uint32_t hi = __reduce_max_sync(0xFFFFFFFFu, (uint32_t)(best >> 32));
    const uint32_t lo = __reduce_max_sync(0xFFFFFFFFu, (uint32_t)(best >> 32) == hi ? (uint32_t)best : 0u);
    const int e = (int)(0xFFFFFFFFu - lo);
    if (lane == j) {
      my_e = e;
      my_l = key_float(hi);
    }
    // the chosen key leaves the set: a select on every word (a conditional
    // store here would be turned back into an indexed store, which puts
    // the whole array in local memory)
    const int qe = (e & 31) == lane ? (e >> 5) : -1;
#pragma unroll
    for (int q = 0; q < NQ; ++q) key[q] = q == qe ? 0ull : key[q];
  }
  const float l0 = __shfl_sync(0xFFFFFFFFu, my_l, 0);
  const float p = lane < k ? expf(my_l - l0) : 0.f;
  float sum = 0.f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xFFFFFFFFu, p, j);
  if (lane < k) {
    idx_row[lane] = my_e;
    w_row[lane] = p / sum;
  }
}

}  // namespace moe

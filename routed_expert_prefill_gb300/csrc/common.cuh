// Internal helpers shared by the library's CUDA translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <utility>

#include "../../include/moe.h"

namespace moe {

// ---------------------------------------------------------------------------
// Device-side status flags (first 256 bytes of every workspace).
// ---------------------------------------------------------------------------
enum : uint32_t {
  FLAG_BAD_EXPERT = 1u << 0,  // an expert id outside [0, E)
  FLAG_BAD_ROW = 1u << 1,     // a CSR row index outside [0, t)
  FLAG_BAD_OFFSETS = 1u << 2, // CSR offsets not monotone / out of range
  FLAG_ROUTE_BOUND = 1u << 3, // a router score left its error bound
  FLAG_TIMEOUT = 1u << 8,     // a bounded device wait gave up
};

struct DeviceStatus {
  uint32_t flags;
  uint32_t timeout_site;  // which wait gave up (kernel-specific code)
  uint32_t route_audit;   // router: largest |score - logit| / bound seen (fp32 bits)
  uint32_t route_cands;   // router: logits recomputed exactly
  uint32_t route_done;    // router, small t: CTAs finished (the last one resets it)
  uint32_t gv_done;       // small-t down kernel: CTAs finished (the last one finalises and resets it)
  uint32_t fused_bar;     // fused decode launch: grid-barrier arrivals (every call adds the grid size)
  uint32_t stall;         // test hook (moe_debug_stall): MOE_STALL_* bits of waits that must run out
  uint32_t pad[56];
};

__device__ __forceinline__ void raise_flag(DeviceStatus* st, uint32_t f) {
  if (st) atomicOr(&st->flags, f);
}

// ---------------------------------------------------------------------------
// bf16 / fp16 bit helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ float bf16f(uint16_t v) { return __uint_as_float(((uint32_t)v) << 16); }

__device__ __forceinline__ uint16_t f2bf(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&b);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// fp16 bits -> bf16 (round to nearest even) as a packed pair replicated:
// scale/bias prepared for the bf16 fma dequantisation.
__device__ __forceinline__ __nv_bfloat16 h2bf(uint16_t hbits) {
  __half hv = *reinterpret_cast<__half*>(&hbits);
  return __float2bfloat16_rn(__half2float(hv));
}

// Dequantise 8 packed 4-bit codes (one 32-bit word, low nibble = even K) to
// 8 bf16 values, w = fma(q, s, b) in bf16 (single rounding), s and b already
// rounded to bf16.  Returns 4 packed bf16x2 words in K order.
__device__ __forceinline__ void dequant8(uint32_t word, __nv_bfloat162 s2, __nv_bfloat162 b2,
                                         uint32_t out[4]) {
  // 0x4300 | q is the bf16 number 128 + q (exact for q < 128).
  const uint32_t MAGIC = 0x43004300u;
  const __nv_bfloat162 k128 = __floats2bfloat162_rn(128.f, 128.f);
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    // byte p holds K = 2p (low nibble) and 2p+1 (high nibble)
    uint32_t b = (word >> (8 * p)) & 0xFFu;
    uint32_t v = ((b & 0xFu) | ((b >> 4) << 16)) | MAGIC;
    __nv_bfloat162 q = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&v), k128);
    __nv_bfloat162 w = __hfma2(q, s2, b2);
    out[p] = *reinterpret_cast<uint32_t*>(&w);
  }
}

// silu(g) * u = g * u * sigmoid(g), sigmoid(g) = (1 + tanh(g / 2)) / 2, with
// the hardware tanh approximation (one special-function op per element;
// absolute error of the sigmoid about 2^-12, below the bf16 rounding of the
// hidden activations it produces).
__device__ __forceinline__ float silu_mul_fast(float g, float u) {
  float th;
  asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(0.5f * g));
  return g * u * fmaf(0.5f, th, 0.5f);
}

// ---------------------------------------------------------------------------
// Workspace layout (host side computes it; kernels receive raw pointers)
// ---------------------------------------------------------------------------
struct WsLayout {
  size_t status;        // DeviceStatus
  size_t csr_rank;      // int32 [t*k]
  size_t csr_counts;    // int32 [nchunks][E]
  size_t csr_base;      // int32 [nchunks][E]
  size_t route;         // router scores and norms (tensor-core router)
  size_t acc;           // float [t][h]
  size_t hg;            // bf16 [t*k][inter]
  size_t hgs;           // bf16 [t][shared_inter]
  size_t ybuf;          // float [t*k][h] (deterministic only)
  size_t xg;            // bf16 gathered token images (packed-weight path only)
  size_t sched;         // scheduler state (counters, tile lists)
  size_t gvpart;        // small-t gate/up partial sums (t <= 16 only)
  size_t fused;         // fused decode launch: logits, gate/up sums, accumulator, counters (t <= 16 only)
  size_t total;
};

constexpr int CSR_CHUNK = 1024;  // pairs per CSR ranking block

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

WsLayout ws_layout(const moe_dims& d, uint32_t flags);

// Raise a kernel's dynamic shared-memory limit once per (kernel, device): the
// attribute is per device and a process may drive several GPUs.  The table is
// keyed by the kernel's address, so template instances that share a signature
// are tracked apart; a later call asking for more bytes sets the limit again.
inline cudaError_t smem_limit_once(const void* kernel, int bytes) {
  struct Entry {
    const void* kernel;
    int dev;
    int bytes;
  };
  static std::mutex mu;
  static Entry table[512];
  static int used = 0;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(mu);
  int slot = -1;
  for (int i = 0; i < used; ++i)
    if (table[i].kernel == kernel && table[i].dev == dev) {
      if (table[i].bytes >= bytes) return cudaSuccess;
      slot = i;
      break;
    }
  err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err != cudaSuccess) return err;
  if (slot < 0 && used < 512) slot = used++;
  if (slot >= 0) table[slot] = Entry{kernel, dev, bytes};
  return cudaSuccess;
}

template <typename Kernel>
cudaError_t set_smem_limit_once(Kernel* kernel, int bytes) {
  return smem_limit_once(reinterpret_cast<const void*>(kernel), bytes);
}

// SM count of the current device, queried once per device.
inline int sm_count() {
  static int n[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 148;
  if (!n[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n[dev] = v > 0 ? v : 148;
  }
  return n[dev];
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of the path is launched with
// programmatic stream serialisation, so it may be launched while the previous
// kernel on the stream is still running.  Each kernel first waits for the
// previous grid to complete with its memory visible (pdl_wait), before any
// other work -- TMEM allocation included, so that a waiting grid never holds
// columns its predecessor still needs -- and then signals that its own
// dependents may launch (pdl_trigger).  What overlaps is the launch and CTA
// rasterisation of the next kernel with the tail of the current one.  Every
// CTA waits before it can exit, so completion stays transitive along the
// stream.  Without the launch attribute both are no-ops.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Thread-local error message (moe_api.cu)
int set_error(int status, const char* fmt, ...);

// Launch accounting (profile.cu): no-ops unless moe_profile_enable(1).
void prof_begin(const char* name, cudaStream_t s);
void prof_end(cudaStream_t s);
#define MOE_LAUNCH(name, stream, ...)  \
  do {                                 \
    ::moe::prof_begin(name, stream);   \
    __VA_ARGS__;                       \
    ::moe::prof_end(stream);           \
  } while (0)

}  // namespace moe

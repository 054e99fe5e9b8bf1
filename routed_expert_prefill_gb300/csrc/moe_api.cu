// The C ABI (include/moe.h): argument checks, workspace layout, dispatch.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>

#include "common.cuh"
#include "experts.cuh"
#include "residency.cuh"

namespace moe {

cudaError_t launch_route_topk(const uint16_t* x, const uint16_t* wr, const float* rbias, int t, int h,
                              int E, int k, int32_t* idx, float* w, float* logits, cudaStream_t stream);
size_t route_smem_bytes(int h, int E);
size_t route_ws_bytes(int t, int h, int E);
cudaError_t launch_route_tc(const uint16_t* x, const uint16_t* wr, const float* rbias, int t, int h, int E, int k,
                            int32_t* idx, float* w, unsigned char* scratch, DeviceStatus* st, cudaStream_t stream,
                            const moe_csr* co = nullptr);
bool route_builds_csr(int t);
cudaError_t launch_build_csr(const int32_t* idx, const float* w, int t, int k, int E, const moe_csr& csr,
                             unsigned char* ws, const WsLayout& L, cudaStream_t stream);
cudaError_t launch_experts_tc(const ExpertsArgs& a, bool deterministic, cudaStream_t stream);
size_t tc_sched_bytes(const moe_dims& d);
size_t packed_max_tiles(const moe_dims& d);
size_t packed_record_bytes(int h, int I, int bits);
size_t packed_pad_rows(const moe_dims& d);
cudaError_t launch_pack(const uint8_t* codes, const uint16_t* scales, const uint16_t* biases, int h, int I,
                        int nrec, int bits, uint8_t* dst, cudaStream_t stream);
cudaError_t launch_experts_packed(const ExpertsArgs& a, const uint8_t* packed, const uint8_t* s_packed,
                                  uint16_t* xg, bool deterministic, cudaStream_t stream,
                                  const PackedBatch* pb = nullptr);
cudaError_t launch_experts_gemv(const ExpertsArgs& a, bool packed, bool deterministic, cudaStream_t stream);
size_t gemv_part_bytes(const moe_dims& d);
bool decode_fused_ok(const moe_dims& d, uint32_t flags);
size_t decode_fused_ws_bytes(const moe_dims& d);
cudaError_t launch_decode_fused(const uint16_t* x, const uint16_t* wr, const float* rbias, const moe_dims& d,
                                const uint8_t* packed, const uint8_t* s_packed, const uint16_t* s_gate, int32_t* idx,
                                float* w, const moe_csr& csr, uint16_t* out, unsigned char* scratch,
                                DeviceStatus* st, cudaStream_t stream);

// Chunks of at most SMALL_T_MAX rows whose (expert, 128-row tile) units are
// few (t * k * inter / 128 below SMALL_T_UNITS on packed records,
// SMALL_T_UNITS_ROWMAJOR on row-major ones) take the weight-streaming
// small-t kernels, unless MOE_FORCE_LARGE_T.  With more units the
// tensor-core kernels are faster: their only per-weight work is the
// dequantisation, where the CUDA-core dot products of the streaming kernels
// cost several more instructions per weight and row.  Graph-timed steps on
// packed records on a GB300: h2048 inter768 E128 k8, t = 1 (48 units)
// 36.0 us streaming against 40.1 on the tensor cores, t = 2 (96) 48.3
// against 42.1, t = 3 (144) 68.6 against 48.3; h4096 inter1536 E256 k8,
// t = 1 (96 units) 91.3 against 58.5.  The row-major tensor-core kernels
// gather token rows with four-row TMA loads and keep the threshold of one
// unit per SM.
constexpr int SMALL_T_MAX = 16;
constexpr int SMALL_T_UNITS = 64;
constexpr int SMALL_T_UNITS_ROWMAJOR = 152;

// Scheduler scratch: room for the larger of the two tensor-core paths' tile
// lists (the packed path's, on its smallest tiles, or the row-major path's).
size_t experts_sched_bytes(const moe_dims& d) {
  const size_t mt = packed_max_tiles(d);
  const int fmax = (d.inter > d.shared_inter ? d.inter : d.shared_inter) / 128;
  const size_t packed = 64 + mt * 16 + mt * fmax * 4 + (size_t)d.t * 4 + 256;
  const size_t rowmajor = tc_sched_bytes(d);
  return packed > rowmajor ? packed : rowmajor;
}

static thread_local char g_err[512] = "";

int set_error(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return status;
}

WsLayout ws_layout(const moe_dims& d, uint32_t flags) {
  WsLayout L{};
  const size_t n = (size_t)d.t * d.k;
  const size_t nchunks = (n + CSR_CHUNK - 1) / CSR_CHUNK;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.status = take(sizeof(DeviceStatus));
  L.csr_rank = take(n * 4);
  L.csr_counts = take(nchunks * d.E * 4);
  L.csr_base = take(nchunks * d.E * 4);
  L.route = take(route_ws_bytes(d.t, d.h, d.E));
  L.acc = take((size_t)d.t * d.h * 4);
  const size_t kmax = d.inter > d.shared_inter ? d.inter : d.shared_inter;
  size_t hg_bytes = n * d.inter * 2;
  if (flags & MOE_PACKED_WEIGHTS) {
    const size_t pb = packed_pad_rows(d) * kmax * 2;
    if (pb > hg_bytes) hg_bytes = pb;
  }
  L.hg = take(hg_bytes);
  L.hgs = take((size_t)d.t * d.shared_inter * 2);
  L.ybuf = (flags & MOE_DETERMINISTIC) ? take(n * d.h * 4) : off;
  L.xg = (flags & MOE_PACKED_WEIGHTS) ? take(packed_pad_rows(d) * d.h * 2) : off;
  L.sched = take(experts_sched_bytes(d));
  L.gvpart = take(gemv_part_bytes(d));
  L.fused = take(d.t <= SMALL_T_MAX ? decode_fused_ws_bytes(d) : 0);
  L.total = off;
  return L;
}

}  // namespace moe

using namespace moe;

namespace {

int dims_bits(const moe_dims* d) { return d->bits ? d->bits : 4; }

int check_dims(const moe_dims* d) {
  if (!d) return set_error(MOE_EINVAL, "dims is NULL");
  if (d->t < 1 || d->t > 65536) return set_error(MOE_ESHAPE, "t=%d outside [1, 65536]", d->t);
  if (d->h < 128 || d->h > 16384 || d->h % 128)
    return set_error(MOE_ESHAPE, "h=%d must be a multiple of 128 in [128, 16384]", d->h);
  if (d->inter < 128 || d->inter > 16384 || d->inter % 128)
    return set_error(MOE_ESHAPE, "inter=%d must be a multiple of 128 in [128, 16384]", d->inter);
  if (d->shared_inter < 0 || d->shared_inter > 16384 || d->shared_inter % 128)
    return set_error(MOE_ESHAPE, "shared_inter=%d must be 0 or a multiple of 128 up to 16384",
                     d->shared_inter);
  if (d->E < 1 || d->E > 1024) return set_error(MOE_ESHAPE, "E=%d outside [1, 1024]", d->E);
  if (d->k < 1 || d->k > 16 || d->k > d->E)
    return set_error(MOE_ESHAPE, "k=%d outside [1, min(E, 16)]", d->k);
  if (d->bits != 0 && d->bits != 2 && d->bits != 3 && d->bits != 4 && d->bits != 8)
    return set_error(MOE_ESHAPE, "bits=%d: the expert records hold 2-, 3-, 4- or 8-bit codes (0 means 4)", d->bits);
  return MOE_OK;
}

int check_ptr(const void* p, const char* name, size_t align, bool nullable = false) {
  if (!p) return nullable ? MOE_OK : set_error(MOE_EINVAL, "%s is NULL", name);
  if ((uintptr_t)p % align) return set_error(MOE_EINVAL, "%s is not %zu-byte aligned", name, align);
  return MOE_OK;
}

int check_ws(const moe_dims* d, uint32_t flags, void* ws, size_t ws_bytes) {
  if (!ws) return set_error(MOE_EWORKSPACE, "workspace is NULL");
  if ((uintptr_t)ws % 256) return set_error(MOE_EWORKSPACE, "workspace is not 256-byte aligned");
  const size_t need = ws_layout(*d, flags).total;
  if (ws_bytes < need)
    return set_error(MOE_EWORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  return MOE_OK;
}

int cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return MOE_OK;
  return set_error(MOE_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define TRY(expr)            \
  do {                       \
    int _s = (expr);         \
    if (_s != MOE_OK) return _s; \
  } while (0)

}  // namespace

__global__ void set_stall_kernel(DeviceStatus* st, uint32_t what) { st->stall = what; }

extern "C" {

const char* moe_last_error(void) { return g_err; }

const char* moe_status_string(int s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_EINVAL: return "MOE_EINVAL";
    case MOE_ESHAPE: return "MOE_ESHAPE";
    case MOE_EWORKSPACE: return "MOE_EWORKSPACE";
    case MOE_ECUDA: return "MOE_ECUDA";
    case MOE_EDEVICE: return "MOE_EDEVICE";
    case MOE_ETIMEOUT: return "MOE_ETIMEOUT";
    default: return "MOE_UNKNOWN";
  }
}

size_t moe_workspace_bytes(const moe_dims* dims, uint32_t flags) {
  if (check_dims(dims) != MOE_OK) return 0;
  return ws_layout(*dims, flags).total;
}

int moe_route_topk(const uint16_t* x, const uint16_t* wr, const float* rbias, const moe_dims* dims,
                   int32_t* idx, float* w, float* logits, void* ws, size_t ws_bytes, void* stream) {
  TRY(check_dims(dims));
  TRY(check_ptr(x, "x", 16));
  TRY(check_ptr(wr, "wr", 16));
  TRY(check_ptr(rbias, "rbias", 4, true));
  TRY(check_ptr(idx, "idx", 4));
  TRY(check_ptr(w, "w", 4));
  TRY(check_ptr(logits, "logits", 4, true));
  if (ws && !logits) {
    TRY(check_ws(dims, 0, ws, ws_bytes));
    const WsLayout L = ws_layout(*dims, 0);
    unsigned char* wsb = (unsigned char*)ws;
    return cuda_status(launch_route_tc(x, wr, rbias, dims->t, dims->h, dims->E, dims->k, idx, w, wsb + L.route,
                                       (DeviceStatus*)(wsb + L.status), (cudaStream_t)stream),
                       "moe_route_topk launch");
  }
  if (route_smem_bytes(dims->h, dims->E) > 227 * 1024)
    return set_error(MOE_ESHAPE, "router tile for h=%d, E=%d exceeds shared memory", dims->h, dims->E);
  return cuda_status(launch_route_topk(x, wr, rbias, dims->t, dims->h, dims->E, dims->k, idx, w, logits,
                                       (cudaStream_t)stream),
                     "moe_route_topk launch");
}

int moe_build_csr(const int32_t* idx, const float* w, const moe_dims* dims, const moe_csr* csr, void* ws,
                  size_t ws_bytes, void* stream) {
  TRY(check_dims(dims));
  TRY(check_ptr(idx, "idx", 4));
  TRY(check_ptr(w, "w", 4));
  if (!csr) return set_error(MOE_EINVAL, "csr is NULL");
  TRY(check_ptr(csr->offsets, "csr->offsets", 4));
  TRY(check_ptr(csr->rows, "csr->rows", 4));
  TRY(check_ptr(csr->weights, "csr->weights", 4));
  TRY(check_ptr(csr->slot_of, "csr->slot_of", 4));
  TRY(check_ws(dims, 0, ws, ws_bytes));
  const WsLayout L = ws_layout(*dims, 0);
  return cuda_status(launch_build_csr(idx, w, dims->t, dims->k, dims->E, *csr, (unsigned char*)ws, L,
                                      (cudaStream_t)stream),
                     "moe_build_csr launch");
}

int moe_route_csr(const uint16_t* x, const uint16_t* wr, const float* rbias, const moe_dims* dims, int32_t* idx,
                  float* w, const moe_csr* csr, void* ws, size_t ws_bytes, void* stream) {
  TRY(check_dims(dims));
  TRY(check_ptr(x, "x", 16));
  TRY(check_ptr(wr, "wr", 16));
  TRY(check_ptr(rbias, "rbias", 4, true));
  TRY(check_ptr(idx, "idx", 4));
  TRY(check_ptr(w, "w", 4));
  if (!csr) return set_error(MOE_EINVAL, "csr is NULL");
  TRY(check_ptr(csr->offsets, "csr->offsets", 4));
  TRY(check_ptr(csr->rows, "csr->rows", 4));
  TRY(check_ptr(csr->weights, "csr->weights", 4));
  TRY(check_ptr(csr->slot_of, "csr->slot_of", 4));
  TRY(check_ws(dims, 0, ws, ws_bytes));
  const WsLayout L = ws_layout(*dims, 0);
  unsigned char* wsb = (unsigned char*)ws;
  const bool fused = route_builds_csr(dims->t);
  TRY(cuda_status(launch_route_tc(x, wr, rbias, dims->t, dims->h, dims->E, dims->k, idx, w, wsb + L.route,
                                  (DeviceStatus*)(wsb + L.status), (cudaStream_t)stream, fused ? csr : nullptr),
                  "moe_route_csr launch"));
  if (fused) return MOE_OK;
  return cuda_status(launch_build_csr(idx, w, dims->t, dims->k, dims->E, *csr, wsb, L, (cudaStream_t)stream),
                     "moe_route_csr launch");
}

// The expert kernels' arguments for one call (pointers already checked).
static ExpertsArgs experts_args(const uint16_t* x, const moe_csr* csr, const moe_qweights* experts,
                                const moe_shared* shared, uint16_t* out, const moe_dims* dims, uint32_t flags,
                                unsigned char* wsb, const WsLayout& L) {
  ExpertsArgs a{};
  a.x = x;
  a.t = dims->t;
  a.h = dims->h;
  a.I = dims->inter;
  a.Is = dims->shared_inter;
  a.E = dims->E;
  a.k = dims->k;
  a.n_pairs = dims->t * dims->k;
  a.offsets = csr->offsets;
  a.rows = csr->rows;
  a.weights = csr->weights;
  a.slot_of = csr->slot_of;
  a.codes = experts ? experts->codes : nullptr;
  a.scales = experts ? experts->scales : nullptr;
  a.biases = experts ? experts->biases : nullptr;
  a.bits = dims_bits(dims);
  a.rec_bytes = (size_t)3 * dims->inter * dims->h * a.bits / 8;
  a.rec_groups = (size_t)3 * dims->inter * dims->h / 64;
  if (dims->shared_inter > 0) {
    a.s_codes = shared->codes;
    a.s_scales = shared->scales;
    a.s_biases = shared->biases;
    a.s_gate = shared->gate;
  }
  a.acc = (float*)(wsb + L.acc);
  a.hg = (uint16_t*)(wsb + L.hg);
  a.hgs = (uint16_t*)(wsb + L.hgs);
  a.ybuf = (flags & MOE_DETERMINISTIC) ? (float*)(wsb + L.ybuf) : nullptr;
  a.sched = wsb + L.sched;
  a.gvpart = gemv_part_bytes(*dims) ? (float*)(wsb + L.gvpart) : nullptr;
  a.status = (DeviceStatus*)(wsb + L.status);
  a.out = out;
  return a;
}

static int check_flags(uint32_t flags) {
  const uint32_t known =
      MOE_DETERMINISTIC | MOE_FORCE_SMALL_T | MOE_FORCE_LARGE_T | MOE_SIMPLE_KERNELS | MOE_PACKED_WEIGHTS |
      MOE_FUSED_DECODE;
  if (flags & ~known) return set_error(MOE_EINVAL, "unknown flag bits 0x%x", flags & ~known);
  if ((flags & MOE_FORCE_SMALL_T) && (flags & MOE_FORCE_LARGE_T))
    return set_error(MOE_EINVAL, "MOE_FORCE_SMALL_T and MOE_FORCE_LARGE_T are exclusive");
  if ((flags & MOE_PACKED_WEIGHTS) && (flags & MOE_SIMPLE_KERNELS))
    return set_error(MOE_EINVAL, "MOE_SIMPLE_KERNELS reads row-major weights, not MOE_PACKED_WEIGHTS");
  return MOE_OK;
}

int moe_experts_fwd(const uint16_t* x, const moe_csr* csr, const moe_qweights* experts,
                    const moe_shared* shared, uint16_t* out, const moe_dims* dims, uint32_t flags, void* ws,
                    size_t ws_bytes, void* stream) {
  TRY(check_dims(dims));
  TRY(check_flags(flags));
  const bool packed = (flags & MOE_PACKED_WEIGHTS) != 0;
  TRY(check_ptr(x, "x", 16));
  TRY(check_ptr(out, "out", 16));
  if (!csr) return set_error(MOE_EINVAL, "csr is NULL");
  TRY(check_ptr(csr->offsets, "csr->offsets", 4));
  TRY(check_ptr(csr->rows, "csr->rows", 4));
  TRY(check_ptr(csr->weights, "csr->weights", 4));
  TRY(check_ptr(csr->slot_of, "csr->slot_of", 4));
  if (!experts) return set_error(MOE_EINVAL, "experts is NULL");
  TRY(check_ptr(experts->codes, "experts->codes", 16));
  TRY(check_ptr(experts->scales, "experts->scales", 16, packed));
  TRY(check_ptr(experts->biases, "experts->biases", 16, packed));
  if (dims->shared_inter > 0) {
    if (!shared) return set_error(MOE_EINVAL, "shared is NULL but shared_inter > 0");
    TRY(check_ptr(shared->codes, "shared->codes", 16));
    TRY(check_ptr(shared->scales, "shared->scales", 16, packed));
    TRY(check_ptr(shared->biases, "shared->biases", 16, packed));
    TRY(check_ptr(shared->gate, "shared->gate", 16, true));
  }
  TRY(check_ws(dims, flags, ws, ws_bytes));
  const WsLayout L = ws_layout(*dims, flags);
  unsigned char* wsb = (unsigned char*)ws;
  const ExpertsArgs a = experts_args(x, csr, experts, shared, out, dims, flags, wsb, L);

  cudaStream_t s = (cudaStream_t)stream;
  if (a.bits != 4 && (!packed || (flags & MOE_FORCE_SMALL_T)))
    return set_error(MOE_EINVAL, "%d-bit records need MOE_PACKED_WEIGHTS and the tensor-core kernels "
                     "(not MOE_FORCE_SMALL_T)", a.bits);
  const bool small_t =
      a.bits == 4 && !(flags & (MOE_FORCE_LARGE_T | MOE_SIMPLE_KERNELS)) &&
      ((flags & MOE_FORCE_SMALL_T) ||
       (dims->t <= SMALL_T_MAX &&
        (long)dims->t * dims->k * (dims->inter / 128) < (packed ? SMALL_T_UNITS : SMALL_T_UNITS_ROWMAJOR)));
  if (small_t)
    return cuda_status(launch_experts_gemv(a, packed, (flags & MOE_DETERMINISTIC) != 0, s), "moe_experts_fwd launch");
  if (packed)
    return cuda_status(launch_experts_packed(a, experts->codes, dims->shared_inter > 0 ? shared->codes : nullptr,
                                             (uint16_t*)(wsb + L.xg), (flags & MOE_DETERMINISTIC) != 0, s),
                       "moe_experts_fwd launch");
  if (flags & MOE_SIMPLE_KERNELS)
    return cuda_status(launch_experts_simple(a, (flags & MOE_DETERMINISTIC) != 0, s), "moe_experts_fwd launch");
  return cuda_status(launch_experts_tc(a, (flags & MOE_DETERMINISTIC) != 0, s), "moe_experts_fwd launch");
}

int moe_forward(const uint16_t* x, const uint16_t* wr, const float* rbias, const moe_qweights* experts,
                const moe_shared* shared, const moe_dims* dims, uint32_t flags, int32_t* idx, float* w,
                const moe_csr* csr, uint16_t* out, void* ws, size_t ws_bytes, void* stream) {
  TRY(check_dims(dims));
  TRY(check_flags(flags));
  if (!(decode_fused_ok(*dims, flags))) {
    TRY(moe_route_csr(x, wr, rbias, dims, idx, w, csr, ws, ws_bytes, stream));
    return moe_experts_fwd(x, csr, experts, shared, out, dims, flags, ws, ws_bytes, stream);
  }
  // the fused decode launch: the same argument checks as the two calls
  TRY(check_ptr(x, "x", 16));
  TRY(check_ptr(wr, "wr", 16));
  TRY(check_ptr(rbias, "rbias", 4, true));
  TRY(check_ptr(idx, "idx", 4));
  TRY(check_ptr(w, "w", 4));
  TRY(check_ptr(out, "out", 16));
  if (!csr) return set_error(MOE_EINVAL, "csr is NULL");
  TRY(check_ptr(csr->offsets, "csr->offsets", 4));
  TRY(check_ptr(csr->rows, "csr->rows", 4));
  TRY(check_ptr(csr->weights, "csr->weights", 4));
  TRY(check_ptr(csr->slot_of, "csr->slot_of", 4));
  if (!experts) return set_error(MOE_EINVAL, "experts is NULL");
  TRY(check_ptr(experts->codes, "experts->codes", 16));
  if (dims->shared_inter > 0) {
    if (!shared) return set_error(MOE_EINVAL, "shared is NULL but shared_inter > 0");
    TRY(check_ptr(shared->codes, "shared->codes", 16));
    TRY(check_ptr(shared->gate, "shared->gate", 16, true));
  }
  TRY(check_ws(dims, flags, ws, ws_bytes));
  const WsLayout L = ws_layout(*dims, flags);
  unsigned char* wsb = (unsigned char*)ws;
  return cuda_status(
      launch_decode_fused(x, wr, rbias, *dims, experts->codes, dims->shared_inter > 0 ? shared->codes : nullptr,
                          dims->shared_inter > 0 ? shared->gate : nullptr, idx, w, *csr, out, wsb + L.fused,
                          (DeviceStatus*)(wsb + L.status), (cudaStream_t)stream),
      "moe_forward launch");
}

int moe_forward_streamed(const uint16_t* x, const uint16_t* wr, const float* rbias, const uint8_t* host_records,
                         const uint8_t* host_miss_records, uint8_t* slots, const moe_shared* shared,
                         const moe_dims* dims, uint32_t flags, int32_t* idx, float* w, const moe_csr* csr,
                         uint16_t* out, void* ws, size_t ws_bytes, moe_streamer* st, void* stream,
                         moe_stream_stats* stats) {
  TRY(check_dims(dims));
  if (!st) return set_error(MOE_EINVAL, "streamer is NULL");
  if (flags & ~(MOE_PACKED_WEIGHTS | MOE_DETERMINISTIC | MOE_FORCE_LARGE_T))
    return set_error(MOE_EINVAL, "flags 0x%x: moe_forward_streamed takes MOE_PACKED_WEIGHTS and MOE_DETERMINISTIC",
                     flags);
  if (!(flags & MOE_PACKED_WEIGHTS)) return set_error(MOE_EINVAL, "moe_forward_streamed needs MOE_PACKED_WEIGHTS");
  const moe_dims& sd = st->dims;
  if (dims->E != sd.E || dims->h != sd.h || dims->inter != sd.inter || dims_bits(dims) != dims_bits(&sd))
    return set_error(MOE_ESHAPE, "dims (E=%d h=%d inter=%d bits=%d) differ from the streamer's (%d %d %d %d)",
                     dims->E, dims->h, dims->inter, dims_bits(dims), sd.E, sd.h, sd.inter, dims_bits(&sd));
  int dev = -1;
  TRY(cuda_status(cudaGetDevice(&dev), "cudaGetDevice"));
  if (dev != st->device)
    return set_error(MOE_EINVAL, "the streamer serves device %d, the current device is %d", st->device, dev);
  // a miss store of another width puts the ring in a region of its own
  const int base_bits = dims_bits(dims);
  const bool split = st->miss_bits != base_bits;
  TRY(check_ptr(host_records, "host_records", 16));
  if (split) TRY(check_ptr(host_miss_records, "host_miss_records", 16));
  if (!split) host_miss_records = host_records;
  TRY(check_ptr(slots, "slots", 16));
  TRY(check_ptr(out, "out", 16));
  if (dims->shared_inter > 0) {
    if (!shared) return set_error(MOE_EINVAL, "shared is NULL but shared_inter > 0");
    TRY(check_ptr(shared->codes, "shared->codes", 16));
    TRY(check_ptr(shared->gate, "shared->gate", 16, true));
  }
  TRY(check_ws(dims, flags, ws, ws_bytes));
  cudaStream_t s = (cudaStream_t)stream;
  // the call follows the previous call on this streamer, on whatever
  // stream that one ran (its batches read the slots this call refills)
  if (st->call_done_recorded) TRY(cuda_status(cudaStreamWaitEvent(s, st->call_done, 0), "stream wait"));
  // router and grouping: checks the remaining pointers before enqueueing
  TRY(moe_route_csr(x, wr, rbias, dims, idx, w, csr, ws, ws_bytes, stream));

  const int E = dims->E, P = st->cfg.pool_slots, R = st->cfg.ring_slots, lag = R / st->cfg.group;
  const size_t rb = st->rec_bytes, rm = split ? st->miss_bytes : st->rec_bytes;
  uint8_t* ring_base = slots + (size_t)P * rb;
  // after a failure the pool's contents are unknown: empty it, and guess no
  // first fetch batch for the next call
  auto fail = [&](cudaError_t e, const char* what) {
    std::fill(st->pool_expert.begin(), st->pool_expert.end(), -1);
    st->spec_expert.clear();
    st->spec_slot.clear();
    return set_error(MOE_ECUDA, "moe_forward_streamed: %s: %s", what, cudaGetErrorString(e));
  };
  cudaError_t e;
  size_t copied = 0;
  // the source and destination of a copy: pool slots from the base store,
  // ring slots from the miss store, each region with its own record size
  auto src_of = [&](int ex, int slot) {
    return slot < P ? host_records + (size_t)ex * rb : host_miss_records + (size_t)ex * rm;
  };
  auto dst_of = [&](int slot) { return slot < P ? slots + (size_t)slot * rb : ring_base + (size_t)(slot - P) * rm; };
  // one copy per run of consecutive experts bound for consecutive slots of
  // one region, over copies [i, n) of the lists
  auto copy_runs = [&](const int32_t* ex, const int32_t* sl, int i, int n) -> cudaError_t {
    while (i < n) {
      const int e0 = ex[i], s0 = sl[i];
      const size_t bytes = s0 < P ? rb : rm;
      int run = 1;
      while (i + run < n && ex[i + run] == e0 + run && sl[i + run] == s0 + run && (sl[i + run] < P) == (s0 < P))
        ++run;
      cudaError_t r = cudaMemcpyAsync(dst_of(s0), src_of(e0, s0), run * bytes, cudaMemcpyHostToDevice, st->copy);
      if (r != cudaSuccess) return r;
      copied += run * bytes;
      i += run;
    }
    return cudaSuccess;
  };
  // every copy of this call follows the end of the last call, whose kernels
  // read the slots (on its own stream, which need not be this one)
  if (st->call_done_recorded && (e = cudaStreamWaitEvent(st->copy, st->call_done, 0)) != cudaSuccess)
    return fail(e, "copy-stream wait");
  // 0. while the chunk is routed, fetch again the last call's first fetch
  // batch (ring slots only)
  const int n_spec = (int)st->spec_expert.size();
  if (n_spec > 0 && (e = copy_runs(st->spec_expert.data(), st->spec_slot.data(), 0, n_spec)) != cudaSuccess)
    return fail(e, "speculative fetch");
  // 1. the chunk's expert counts on the host
  if ((e = cudaMemcpyAsync(st->h_offsets, csr->offsets, (E + 1) * sizeof(int32_t), cudaMemcpyDeviceToHost, s)) !=
      cudaSuccess)
    return fail(e, "offsets copy");
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return fail(e, "stream sync");
  for (int i = 0; i < E; ++i) {
    const int32_t n = st->h_offsets[i + 1] - st->h_offsets[i];
    st->counts[i] = n > 0 ? n : 0;  // bad offsets: flagged on the device, nothing runs
  }
  // 2. the plan, and the record and batch maps on the device
  moe_residency_plan pl{};
  pl.pool_expert = st->pool_expert.data();
  pl.pool_last = st->pool_last.data();
  pl.rec = st->plan_rec.data();
  pl.batch = st->plan_batch.data();
  pl.copy_expert = st->copy_expert.data();
  pl.copy_slot = st->copy_slot.data();
  pl.wait_for = st->wait_for.data();
  const int ps = plan_residency(st->counts.data(), E, st->cfg, ++st->call, pl);
  if (ps != MOE_OK) {
    std::fill(st->pool_expert.begin(), st->pool_expert.end(), -1);
    return ps;
  }
  // One code width: rec is the record's index in the slot buffer and
  // batch_of its batch.  Two widths: rec counts within the record's region
  // (pool or ring) and batch_of = 2 batch + (ring record), so that each pass
  // of the expert kernels sees one width.  batch_of[E] is the shared expert.
  int32_t* map_rec = st->h_maps;
  int32_t* map_batch = st->h_maps + E;
  std::vector<uint8_t> has_base(pl.n_batches, 0), has_ring(pl.n_batches, 0);
  for (int i = 0; i < E; ++i) {
    const int r = st->plan_rec[i], b = st->plan_batch[i];
    const bool ring = r >= P;
    map_rec[i] = (split && ring) ? r - P : r;
    map_batch[i] = (split && b >= 0) ? 2 * b + (ring ? 1 : 0) : b;
    if (b >= 0) (ring ? has_ring : has_base)[b] = 1;
  }
  map_batch[E] = 0;
  if ((e = cudaMemcpyAsync(st->d_maps, st->h_maps, (2 * E + 1) * sizeof(int32_t), cudaMemcpyHostToDevice, s)) !=
      cudaSuccess)
    return fail(e, "map copy");

  const WsLayout L = ws_layout(*dims, flags);
  unsigned char* wsb = (unsigned char*)ws;
  const ExpertsArgs a = experts_args(x, csr, nullptr, shared, out, dims, flags, wsb, L);
  const bool det = (flags & MOE_DETERMINISTIC) != 0;
  const uint8_t* s_packed = dims->shared_inter > 0 ? shared->codes : nullptr;
  uint16_t* xg = (uint16_t*)(wsb + L.xg);
  // the passes of the expert kernels, in order: per batch, one pass (one
  // width) or, with two widths, a pool pass and/or a ring pass
  struct Pass {
    int batch, filter;
    bool ring;
  };
  std::vector<Pass> passes;
  for (int b = 0; b < pl.n_batches; ++b) {
    if (!split) {
      passes.push_back({b, b, false});
      continue;
    }
    if (b == 0 || has_base[b]) passes.push_back({b, 2 * b, false});
    if (has_ring[b]) passes.push_back({b, 2 * b + 1, true});
  }
  auto run = [&](size_t i) -> cudaError_t {
    const Pass& q = passes[i];
    ExpertsArgs aq = a;
    aq.bits = q.ring ? st->miss_bits : base_bits;
    PackedBatch pb{st->d_maps, split ? (q.ring ? R : P) : P + R, st->d_maps + E, q.filter, i == 0,
                   i + 1 == passes.size()};
    return launch_experts_packed(aq, q.ring ? ring_base : slots, s_packed, xg, det, s, &pb);
  };
  // 3-4. the fetch batches, two events each, and batch 0 (the resident
  // experts and the shared expert, no fetch).  Fetch batch 1 is enqueued
  // first so that the copies start while batch 0's launches are issued.
  // Copies of batch b are the list entries [first[b], first[b + 1]).
  std::vector<int> first(pl.n_batches + 1, pl.n_copies);
  for (int i = pl.n_copies - 1; i >= 0; --i) first[st->plan_batch[pl.copy_expert[i]]] = i;
  for (int b = pl.n_batches - 1; b >= 1; --b) first[b] = std::min(first[b], first[b + 1]);
  // the speculative copies are batch 1 when they match it entry for entry
  bool spec_used = n_spec > 0 && pl.n_batches > 1 && first[2] - first[1] == n_spec;
  for (int i = 0; spec_used && i < n_spec; ++i)
    spec_used = pl.copy_expert[first[1] + i] == st->spec_expert[i] && pl.copy_slot[first[1] + i] == st->spec_slot[i];
  // fetch batch b: wait until the batch that last read its ring slots is
  // done, copy, and signal "fetched"
  auto fetch = [&](int b) -> cudaError_t {
    cudaError_t r;
    if (!(b == 1 && spec_used)) {
      if (pl.wait_for[b] >= 1 &&
          (r = cudaStreamWaitEvent(st->copy, st->done[pl.wait_for[b] % lag], 0)) != cudaSuccess)
        return r;
      if ((r = copy_runs(pl.copy_expert, pl.copy_slot, first[b], first[b + 1])) != cudaSuccess) return r;
    }
    return cudaEventRecord(st->fetched, st->copy);
  };
  size_t pi = 0;
  if (pl.n_batches > 1 && (e = fetch(1)) != cudaSuccess) return fail(e, "record fetch");
  for (; pi < passes.size() && passes[pi].batch == 0; ++pi)
    if ((e = run(pi)) != cudaSuccess) return fail(e, "batch 0");
  for (int b = 1; b < pl.n_batches; ++b) {
    if (b > 1 && (e = fetch(b)) != cudaSuccess) return fail(e, "record fetch");
    if ((e = cudaStreamWaitEvent(s, st->fetched, 0)) != cudaSuccess) return fail(e, "stream wait");
    for (; pi < passes.size() && passes[pi].batch == b; ++pi)
      if ((e = run(pi)) != cudaSuccess) return fail(e, "batch");
    if ((e = cudaEventRecord(st->done[b % lag], s)) != cudaSuccess) return fail(e, "event record");
  }
  if ((e = cudaEventRecord(st->call_done, s)) != cudaSuccess) return fail(e, "event record");
  st->call_done_recorded = true;
  // the guess for the next call: this call's first fetch batch, when it
  // holds ring records only
  st->spec_expert.clear();
  st->spec_slot.clear();
  if (pl.n_batches > 1) {
    bool ring_only = true;
    for (int i = first[1]; i < first[2]; ++i) ring_only = ring_only && pl.copy_slot[i] >= P;
    if (ring_only)
      for (int i = first[1]; i < first[2]; ++i) {
        st->spec_expert.push_back(pl.copy_expert[i]);
        st->spec_slot.push_back(pl.copy_slot[i]);
      }
  }
  if (stats) {
    stats->resident = 0;
    stats->filled = 0;
    for (int i = 0; i < E; ++i) stats->resident += st->plan_batch[i] == 0;
    for (int i = 0; i < pl.n_copies; ++i) stats->filled += pl.copy_slot[i] < P;
    stats->streamed = pl.n_copies - stats->filled;
    stats->batches = pl.n_batches - 1;
    stats->bytes = (int64_t)copied;
    stats->prefetched = n_spec;
    stats->prefetch_used = spec_used ? 1 : 0;
  }
  return MOE_OK;
}

size_t moe_packed_bytes(const moe_dims* dims, int shared) {
  if (check_dims(dims) != MOE_OK) return 0;
  if (shared) return dims->shared_inter > 0 ? packed_record_bytes(dims->h, dims->shared_inter, dims_bits(dims)) : 0;
  return (size_t)dims->E * packed_record_bytes(dims->h, dims->inter, dims_bits(dims));
}

int moe_pack_experts(const moe_qweights* src, const moe_dims* dims, int shared, void* dst, size_t dst_bytes,
                     void* stream) {
  TRY(check_dims(dims));
  if (!src) return set_error(MOE_EINVAL, "src is NULL");
  TRY(check_ptr(src->codes, "src->codes", 16));
  TRY(check_ptr(src->scales, "src->scales", 2));
  TRY(check_ptr(src->biases, "src->biases", 2));
  TRY(check_ptr(dst, "dst", 16));
  if (shared && dims->shared_inter == 0) return set_error(MOE_ESHAPE, "shared_inter is 0: nothing to pack");
  const size_t need = moe_packed_bytes(dims, shared);
  if (dst_bytes < need) return set_error(MOE_EINVAL, "dst has %zu bytes, needs %zu", dst_bytes, need);
  const int I = shared ? dims->shared_inter : dims->inter;
  return cuda_status(launch_pack(src->codes, src->scales, src->biases, dims->h, I, shared ? 1 : dims->E, dims_bits(dims),
                                 (uint8_t*)dst, (cudaStream_t)stream),
                     "moe_pack_experts launch");
}

int moe_clear_device_status(void* ws, void* stream) {
  if (!ws) return set_error(MOE_EWORKSPACE, "workspace is NULL");
  return cuda_status(cudaMemsetAsync(ws, 0, sizeof(DeviceStatus), (cudaStream_t)stream),
                     "moe_clear_device_status");
}

int moe_debug_stall(void* ws, uint32_t what, void* stream) {
  if (!ws) return set_error(MOE_EWORKSPACE, "workspace is NULL");
  if (what & ~(MOE_STALL_WEIGHT_COPIES | MOE_STALL_GRID_BARRIER))
    return set_error(MOE_EINVAL, "unknown stall bits 0x%x", what & ~(MOE_STALL_WEIGHT_COPIES | MOE_STALL_GRID_BARRIER));
  set_stall_kernel<<<1, 1, 0, (cudaStream_t)stream>>>((DeviceStatus*)ws, what);
  return cuda_status(cudaGetLastError(), "moe_debug_stall");
}

int moe_read_device_status(void* ws, void* stream) {
  if (!ws) return set_error(MOE_EWORKSPACE, "workspace is NULL");
  DeviceStatus st;
  cudaStream_t s = (cudaStream_t)stream;
  TRY(cuda_status(cudaMemcpyAsync(&st, ws, sizeof(st), cudaMemcpyDeviceToHost, s), "status read"));
  TRY(cuda_status(cudaStreamSynchronize(s), "status sync"));
  TRY(cuda_status(cudaMemsetAsync(ws, 0, sizeof(DeviceStatus), s), "status clear"));
  TRY(cuda_status(cudaStreamSynchronize(s), "status clear sync"));
  if (st.flags & FLAG_TIMEOUT)
    return set_error(MOE_ETIMEOUT, "a bounded device wait gave up (site %u)", st.timeout_site);
  if (st.flags & (FLAG_BAD_EXPERT | FLAG_BAD_ROW | FLAG_BAD_OFFSETS | FLAG_ROUTE_BOUND))
    return set_error(MOE_EDEVICE, "device-side check failed (flags 0x%x: %s%s%s%s)", st.flags,
                     (st.flags & FLAG_BAD_EXPERT) ? "expert id out of range " : "",
                     (st.flags & FLAG_BAD_ROW) ? "row out of range " : "",
                     (st.flags & FLAG_BAD_OFFSETS) ? "bad offsets " : "",
                     (st.flags & FLAG_ROUTE_BOUND) ? "router score outside its error bound" : "");
  return MOE_OK;
}

}  // extern "C"

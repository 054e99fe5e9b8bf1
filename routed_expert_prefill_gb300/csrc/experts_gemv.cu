// Small-t expert FFNs (decode-shaped chunks): weight-streaming GEMV kernels
// for cherenkov qwen4_exp, prefill/experts.rs, pf_experts (gate/up quantised
// matmuls -> silu_mul -> down quantised matmul -> scatter_add_rows, plus the
// shared expert), for chunks whose experts see at most a few rows each.
//
// With t rows an expert sees at most t of them, so every weight is used by a
// handful of dot products and the work is bound by the weight bytes.  One
// CTA of 128 threads owns 32 output rows of one (active) expert: four
// threads per weight row, each taking 16 of the 64 K of every chunk, read the
// 4-bit codes straight from HBM (coalesced 8-byte loads), dequantise them
// with the same bf16 fma as the tensor-core path (w = fma(q, s, b), one
// rounding), and accumulate the exact bf16 x bf16 products in fp32 for each
// of the expert's rows (16 at a time).  The four partial sums of a row
// combine as (p0 + p1) + (p2 + p3).
//   gateup: hg[list position][f] = bf16(silu(gate) * up)
//   down:   acc[row][f] += weight * y (fp32 atomics), or, deterministic
//           mode, ybuf[list position][f] = y and the shared expert stores
//           acc[row][f] = gate * y; the finalize pass then sums the list
//           positions of each row in ascending order.
// Both weight layouts are read: the row-major records (moe_qweights) and the
// packed blocks of moe_pack_experts.
//
// Packed weights at t <= 16 take the streaming variant (gv2_*): per CTA one
// thread bulk-copies whole 128-row blocks (codes, scales, biases; 9 KB per
// gate/up chunk, 4.5 KB per down chunk) into a 72 KB shared-memory ring and
// eight warps consume them, two threads per weight row (32 K each), with the
// token rows staged once in shared memory.  gate/up splits K in up to four
// slices when few experts are active, writing fp32 partial sums per slice;
// the down kernel sums the slices in order, applies silu(gate) * up (bf16,
// as the tensor-core path stores it) into shared memory and streams the down
// blocks the same way.
#include "experts.cuh"
#include "tc_ptx.cuh"

namespace moe {

cudaError_t launch_shared_gate(const uint16_t* x, const uint16_t* g, int t, int h, float* out, cudaStream_t stream);

constexpr int GV2_KS_MAX = 8;  // gate/up K slices of the streaming small-t kernels

namespace {

using namespace tc;

constexpr int GV_THREADS = 128;
constexpr int GV_ROWS = 32;  // output rows per CTA
constexpr int GV_RB = 16;    // token rows per pass over the weights (at most)
constexpr int GV_KC = 64;    // K per quantisation group
constexpr int GV_QB = PACK_QB;
// Rows per pass NB is a template parameter (1, 2, 4, 8 or 16: the smallest
// that covers min(t, 16)), so a one-row step runs a short loop: the fully
// unrolled body for 16 rows does not fit the instruction cache.  Weight
// chunks kept in flight per thread:
template <int NB>
__host__ __device__ constexpr int gv_pf() { return NB >= 8 ? 4 : 8; }

struct GvParams {
  int t, h, I, Is, E, k;
  int deterministic, packed;
  const uint16_t* x;
  const int32_t* offsets;
  const int32_t* rows;
  const float* weights;
  const uint8_t* codes;  // routed records (row-major or packed)
  const uint16_t* scales;
  const uint16_t* biases;
  const uint8_t* s_codes;  // shared record
  const uint16_t* s_scales;
  const uint16_t* s_biases;
  const float* gate_vals;  // per-row shared gate or null
  uint16_t* hg;            // bf16 [t*k][I]
  uint16_t* hgs;           // bf16 [t][Is]
  float* acc;              // fp32 [t][h]
  float* ybuf;             // fp32 [t*k][h] (deterministic)
  DeviceStatus* status;
  const int32_t* slot_of;  // [t*k] list position of each (row, slot), -1 if dropped
  uint16_t* out;           // bf16 [t][h]
};

// Where one thread finds its 16 weights of each K chunk of one weight row:
// the codes at code + kc * kstride, the scale and the bias (16-bit) at
// sc + kc * sstride and bi + kc * sstride (byte strides).  Row-major records
// (moe_qweights): the row's codes are contiguous (32 bytes per chunk) and its
// fp16 scales and biases consecutive.  Packed records: chunk kc of a 128-row
// tile is one block (codes, then bf16 scales, then bf16 biases).
struct RowSrc {
  const uint8_t* code;
  const uint8_t* sc;
  const uint8_t* bi;
  uint32_t kstride, sstride;
};

// Row f of matrix `mat` (0 gate, 1 up, 2 down) of expert e (shared: the
// shared record), for quarter `part` of every chunk.
__device__ __forceinline__ RowSrc row_src(const GvParams& P, bool shared, int e, int mat, int f, int part) {
  const int h = P.h, Iu = shared ? P.Is : P.I;
  const int K = mat == 2 ? Iu : h;
  const uint8_t* c = shared ? P.s_codes : P.codes;
  RowSrc R;
  if (P.packed) {
    const uint8_t* rec = c + (shared ? 0 : (size_t)e * packed_rec_bytes(h, Iu));
    const uint8_t* tile;
    if (mat < 2) {  // [128-row tile][K chunk][gate block][up block]
      tile = rec + (size_t)(f / 128) * (h / GV_KC) * 2 * GV_QB + (size_t)mat * GV_QB;
      R.kstride = 2 * GV_QB;
    } else {  // [128-row tile of h][K chunk][block]
      tile = rec + packed_gu_bytes(h, Iu) + (size_t)(f / 128) * (Iu / GV_KC) * GV_QB;
      R.kstride = GV_QB;
    }
    const int o = f % 128;
    R.code = tile + o * 32 + part * 8;
    R.sc = tile + 4096 + o * 2;
    R.bi = tile + 4096 + 256 + o * 2;
    R.sstride = R.kstride;
  } else {
    const size_t mat_bytes = (size_t)Iu * h / 2, mat_groups = (size_t)Iu * h / GV_KC;
    const size_t e_off = shared ? 0 : (size_t)e;
    const uint16_t* s = shared ? P.s_scales : P.scales;
    const uint16_t* b = shared ? P.s_biases : P.biases;
    const size_t g0 = e_off * 3 * mat_groups + (size_t)mat * mat_groups + (size_t)f * (K / GV_KC);
    R.code = c + e_off * 3 * mat_bytes + (size_t)mat * mat_bytes + (size_t)f * (K / 2) + part * 8;
    R.sc = reinterpret_cast<const uint8_t*>(s + g0);
    R.bi = reinterpret_cast<const uint8_t*>(b + g0);
    R.kstride = 32;
    R.sstride = 2;
  }
  return R;
}

// Raw codes, scale and bias of one thread's 16 weights of chunk kc, loaded
// ahead of use; dequant() turns them into 8 bf16 pairs in K order.
struct WRaw {
  uint2 c;
  uint32_t sb;  // scale bits (low half), bias bits (high half); bf16 (packed) or fp16 (row-major)
};

__device__ __forceinline__ WRaw load_raw(const RowSrc& R, int kc) {
  WRaw r;
  r.c = __ldg(reinterpret_cast<const uint2*>(R.code + (size_t)kc * R.kstride));
  const uint32_t sv = __ldg(reinterpret_cast<const uint16_t*>(R.sc + (size_t)kc * R.sstride));
  const uint32_t bv = __ldg(reinterpret_cast<const uint16_t*>(R.bi + (size_t)kc * R.sstride));
  r.sb = sv | (bv << 16);
  return r;
}

__device__ __forceinline__ void dequant(bool packed, const WRaw& r, uint32_t (&out)[8]) {
  if (packed) {
    const uint16_t sbits = (uint16_t)(r.sb & 0xFFFFu), bbits = (uint16_t)(r.sb >> 16);
    const __nv_bfloat16 s = *reinterpret_cast<const __nv_bfloat16*>(&sbits);
    const __nv_bfloat16 b = *reinterpret_cast<const __nv_bfloat16*>(&bbits);
    const __nv_bfloat162 s2 = __halves2bfloat162(s, s), b2 = __halves2bfloat162(b, b);
    const __nv_bfloat162 k128 = __floats2bfloat162_rn(128.f, 128.f);
    const uint32_t w[2] = {r.c.x, r.c.y};
    // packed word: (word >> 4i) & 0x000F000F is the pair (K 2i, K 2i + 1)
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t v = ((w[j] >> (4 * i)) & 0x000F000Fu) | 0x43004300u;
        __nv_bfloat162 q = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&v), k128);
        __nv_bfloat162 o = __hfma2(q, s2, b2);
        out[4 * j + i] = *reinterpret_cast<uint32_t*>(&o);
      }
  } else {
    const __nv_bfloat16 s = h2bf((uint16_t)(r.sb & 0xFFFFu)), b = h2bf((uint16_t)(r.sb >> 16));
    const __nv_bfloat162 s2 = __halves2bfloat162(s, s), b2 = __halves2bfloat162(b, b);
    dequant8(r.c.x, s2, b2, out);
    dequant8(r.c.y, s2, b2, out + 4);
  }
}

// acc[r] += sum over the 16 K of w * a_r, a_r = 16 bf16 of row r (two uint4).
__device__ __forceinline__ void fma16(const uint32_t (&w)[8], const uint4& a0, const uint4& a1, float& acc) {
  const uint32_t a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    acc = fmaf(bf16lo(w[i]), bf16lo(a[i]), acc);
    acc = fmaf(bf16hi(w[i]), bf16hi(a[i]), acc);
  }
}

__device__ __forceinline__ float quad_sum(float v) {
  // (p0 + p1) + (p2 + p3) on every lane of the quad
  v = v + __shfl_xor_sync(0xFFFFFFFFu, v, 1);
  v = v + __shfl_xor_sync(0xFFFFFFFFu, v, 2);
  return v;
}

// The j-th expert (ascending id) with a non-empty list, or -1.
__device__ int find_active(const int32_t* offsets, int E, int j, int* s_e) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int found = -1, seen = 0;
    for (int e0 = 0; e0 < E && found < 0; e0 += 32) {
      const int e = e0 + lane;
      const bool nz = e < E && offsets[e + 1] > offsets[e];
      const uint32_t m = __ballot_sync(0xFFFFFFFFu, nz);
      const int c = __popc(m);
      if (j < seen + c) {
        uint32_t mm = m;
        for (int s = 0; s < j - seen; ++s) mm &= mm - 1;
        found = e0 + __ffs(mm) - 1;
      }
      seen += c;
    }
    if (lane == 0) *s_e = found;
  }
  __syncthreads();
  return *s_e;
}

__device__ __forceinline__ float silu_mul_f(float g, float u) { return silu_mul_fast(g, u); }

// Rows of the unit: routed expert e (its list entries) or the shared expert (all t rows).
struct GvRows {
  int base, n;  // list start (routed) and length
  bool shared;
};

template <bool GATEUP, int NB>
__global__ void __launch_bounds__(GV_THREADS)
gemv_kernel(GvParams P, int groups) {
  pdl_wait();
  pdl_trigger();
  constexpr int GV_PF = gv_pf<NB>();
  __shared__ int s_e;
  __shared__ int s_row[NB];
  __shared__ float s_w[NB];
  const bool shared = blockIdx.y == 1;
  if (GATEUP && blockIdx.y == 0 && (!P.deterministic || P.Is == 0)) {
    // zero the fp32 block accumulator (the down kernel adds into it)
    float4* a4 = reinterpret_cast<float4*>(P.acc);
    const size_t n4 = (size_t)P.t * P.h / 4;
    for (size_t i = (size_t)blockIdx.x * GV_THREADS + threadIdx.x; i < n4; i += (size_t)gridDim.x * GV_THREADS)
      a4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int Iu = shared ? P.Is : P.I;
  const int out_rows = GATEUP ? Iu : P.h;
  const int ng = out_rows / GV_ROWS;
  int e = P.E, g = blockIdx.x;
  GvRows R{0, P.t, true};
  if (shared) {
    if (Iu == 0 || g >= ng) return;
  } else {
    const int j = blockIdx.x / groups;
    g = blockIdx.x % groups;
    if (g >= ng) return;
    e = find_active(P.offsets, P.E, j, &s_e);
    if (e < 0) return;
    R.shared = false;
    R.base = P.offsets[e];
    R.n = P.offsets[e + 1] - R.base;
    if (R.base < 0 || R.n > P.t || R.base + R.n > P.t * P.k) {
      if (threadIdx.x == 0) raise_flag(P.status, FLAG_BAD_OFFSETS);
      return;
    }
  }
  const int rr = threadIdx.x >> 2, part = threadIdx.x & 3;
  const int f = g * GV_ROWS + rr;
  const int K = GATEUP ? P.h : Iu;
  const int nkc = K / GV_KC;
  const bool packed = P.packed != 0;
  const RowSrc S0 = row_src(P, shared, e, GATEUP ? 0 : 2, f, part);
  const RowSrc S1 = row_src(P, shared, e, GATEUP ? 1 : 2, f, part);

  for (int rb = 0; rb < R.n; rb += NB) {
    const int nb = min(NB, R.n - rb);
    __syncthreads();  // s_row / s_w of the previous batch are no longer read
    if (threadIdx.x < nb) {
      const int i = rb + threadIdx.x;
      int row;
      float wv = 1.f;
      if (R.shared) {
        row = i;
        if (P.gate_vals) wv = P.gate_vals[i];
      } else {
        row = P.rows[R.base + i];
        wv = P.weights[R.base + i];
        if (row < 0 || row >= P.t) {
          raise_flag(P.status, FLAG_BAD_ROW);
          row = -1;
        }
      }
      s_row[threadIdx.x] = row;
      s_w[threadIdx.x] = wv;
    }
    __syncthreads();
    float a0[NB], a1[NB];
#pragma unroll
    for (int r = 0; r < NB; ++r) a0[r] = a1[r] = 0.f;
    // GV_PF chunks of weights in flight per thread: chunk kc + GV_PF is
    // requested as chunk kc is consumed
    WRaw q0[GV_PF], q1[GV_PF];
#pragma unroll
    for (int i = 0; i < GV_PF; ++i) {
      if (i < nkc) {
        q0[i] = load_raw(S0, i);
        if (GATEUP) q1[i] = load_raw(S1, i);
      }
    }
    for (int kc0 = 0; kc0 < nkc; kc0 += GV_PF) {
#pragma unroll
      for (int i = 0; i < GV_PF; ++i) {
        const int kc = kc0 + i;
        if (kc < nkc) {
          uint32_t w0[8], w1[8];
          dequant(packed, q0[i], w0);
          if (GATEUP) dequant(packed, q1[i], w1);
          if (kc + GV_PF < nkc) {
            q0[i] = load_raw(S0, kc + GV_PF);
            if (GATEUP) q1[i] = load_raw(S1, kc + GV_PF);
          }
          const int k0 = kc * GV_KC + part * 16;
#pragma unroll
          for (int r = 0; r < NB; ++r) {
            if (r < nb) {
              const uint4* src;
              if (GATEUP) {
                const int row = s_row[r];
                src = reinterpret_cast<const uint4*>(P.x + (size_t)(row < 0 ? 0 : row) * P.h + k0);
              } else {
                src = R.shared ? reinterpret_cast<const uint4*>(P.hgs + (size_t)(rb + r) * P.Is + k0)
                               : reinterpret_cast<const uint4*>(P.hg + (size_t)(R.base + rb + r) * P.I + k0);
              }
              const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
              fma16(w0, v0, v1, a0[r]);
              if (GATEUP) fma16(w1, v0, v1, a1[r]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < NB; ++r) {
      if (r < nb) {
        const float y0 = quad_sum(a0[r]);
        const float y1 = GATEUP ? quad_sum(a1[r]) : 0.f;
        if (part == 0) {
          const int row = s_row[r];
          if (GATEUP) {
            const float hv = row < 0 ? 0.f : silu_mul_f(y0, y1);
            uint16_t* dst = R.shared ? P.hgs + (size_t)(rb + r) * P.Is : P.hg + (size_t)(R.base + rb + r) * P.I;
            dst[f] = f2bf(hv);
          } else if (P.deterministic && !R.shared) {
            P.ybuf[(size_t)(R.base + rb + r) * P.h + f] = y0;
          } else if (row >= 0) {
            float* d = P.acc + (size_t)row * P.h + f;
            if (P.deterministic) *d = s_w[r] * y0;
            else atomicAdd(d, s_w[r] * y0);
          }
        }
      }
    }
  }
}


// ---------------------------------------------------------------------------
// Streaming small-t kernels for packed weights
// ---------------------------------------------------------------------------
constexpr int GV2_CONS = 256;               // consumer threads: 128 rows x 2 halves of K
constexpr int GV2_THREADS = GV2_CONS + 32;  // + one producer warp
constexpr int GV2_RING = 73728;             // bytes of the block ring
constexpr uint64_t GV2_WAIT_NS = 2000000000ull;

struct Gv2Params {
  GvParams p;
  float* part;   // [KS][t*k + t][2][kmax]
  int KS, kmax;
};

__device__ __forceinline__ void gv2_timeout(DeviceStatus* st, volatile int* abort, uint32_t site) {
  if (atomicOr(&st->flags, FLAG_TIMEOUT) == 0) st->timeout_site = site;
  *abort = 1;
}

// 32 weights of one packed-block row (half hf of the chunk), 16 bf16 pairs in K order.
__device__ __forceinline__ void dequant_half(const uint8_t* blk, int o, int hf, uint32_t (&w)[16]) {
  const uint4 c = *reinterpret_cast<const uint4*>(blk + o * 32 + hf * 16);
  const uint16_t sbits = *reinterpret_cast<const uint16_t*>(blk + 4096 + o * 2);
  const uint16_t bbits = *reinterpret_cast<const uint16_t*>(blk + 4096 + 256 + o * 2);
  const __nv_bfloat16 s = *reinterpret_cast<const __nv_bfloat16*>(&sbits);
  const __nv_bfloat16 b = *reinterpret_cast<const __nv_bfloat16*>(&bbits);
  const __nv_bfloat162 s2 = __halves2bfloat162(s, s), b2 = __halves2bfloat162(b, b);
  const __nv_bfloat162 k128 = __floats2bfloat162_rn(128.f, 128.f);
  const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t v = ((cw[j] >> (4 * i)) & 0x000F000Fu) | 0x43004300u;
      __nv_bfloat162 q = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&v), k128);
      __nv_bfloat162 r = __hfma2(q, s2, b2);
      w[4 * j + i] = *reinterpret_cast<uint32_t*>(&r);
    }
}

// acc += sum over 32 K of w * a, a = 32 fp32 in shared memory (16-byte aligned).
__device__ __forceinline__ void fma32f(const uint32_t (&w)[16], const float* a, float& acc) {
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const float4 x = *reinterpret_cast<const float4*>(a + 4 * v);
    acc = fmaf(bf16lo(w[2 * v]), x.x, acc);
    acc = fmaf(bf16hi(w[2 * v]), x.y, acc);
    acc = fmaf(bf16lo(w[2 * v + 1]), x.z, acc);
    acc = fmaf(bf16hi(w[2 * v + 1]), x.w, acc);
  }
}

// acc += sum over 32 K of w * a, a = 32 bf16 in shared memory (16-byte aligned).
__device__ __forceinline__ void fma32(const uint32_t (&w)[16], const uint16_t* a, float& acc) {
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint4 x = *reinterpret_cast<const uint4*>(a + 8 * v);
    const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = fmaf(bf16lo(w[4 * v + i]), bf16lo(xw[i]), acc);
      acc = fmaf(bf16hi(w[4 * v + i]), bf16hi(xw[i]), acc);
    }
  }
}

// Rows of a unit in shared memory: token row, weight (or shared gate) and
// position in the partial / hg arrays.
template <int NB>
struct Gv2Rows {
  int row[NB];
  float w[NB];
  int pos[NB];
  int n;
};

// Unit decode shared by both kernels: returns false if the CTA has no work.
template <int NB>
__device__ bool gv2_unit(const GvParams& P, int units_per_e, int* s_e, Gv2Rows<NB>& R, int& e, int& sub,
                         bool& shared) {
  shared = blockIdx.y == 1;
  if (shared) {
    if (P.Is == 0 || (int)blockIdx.x >= units_per_e) return false;
    e = P.E;
    sub = blockIdx.x;
  } else {
    const int j = blockIdx.x / units_per_e;
    sub = blockIdx.x % units_per_e;
    e = find_active(P.offsets, P.E, j, s_e);
    if (e < 0) return false;
  }
  if (threadIdx.x == 0) {
    int n;
    if (shared) {
      n = P.t;
      for (int i = 0; i < n && i < NB; ++i) {
        R.row[i] = i;
        R.w[i] = P.gate_vals ? P.gate_vals[i] : 1.f;
        R.pos[i] = P.t * P.k + i;
      }
    } else {
      const int base = P.offsets[e];
      n = P.offsets[e + 1] - base;
      if (base < 0 || base + n > P.t * P.k) {
        raise_flag(P.status, FLAG_BAD_OFFSETS);
        n = 0;
      }
      for (int i = 0; i < n && i < NB; ++i) {
        int row = P.rows[base + i];
        if (row < 0 || row >= P.t) {
          raise_flag(P.status, FLAG_BAD_ROW);
          row = -1;
        }
        R.row[i] = row;
        R.w[i] = P.weights[base + i];
        R.pos[i] = base + i;
      }
    }
    if (n > NB) {  // the dispatch keeps every list within NB rows
      raise_flag(P.status, FLAG_BAD_OFFSETS);
      n = NB;
    }
    R.n = n;
  }
  __syncthreads();
  return R.n > 0;
}

// gate/up: unit = (expert, 128-row feature tile rt, K slice ks).
template <int NB>
__global__ void __launch_bounds__(GV2_THREADS, 1) gv2_gateup(Gv2Params Q) {
  pdl_wait();
  pdl_trigger();
  const GvParams& P = Q.p;
  extern __shared__ __align__(16) uint8_t sm[];
  uint8_t* ring = sm;
  constexpr int ST = GV2_RING / (2 * GV_QB);  // 8 stages of one gate+up block pair
  static_assert(ST <= 32, "stage bit masks");
  __shared__ uint64_t full[ST], empty[ST];
  __shared__ int s_e, abort_flag;
  __shared__ Gv2Rows<NB> R;
  if (blockIdx.y == 0 && (!P.deterministic || P.Is == 0)) {
    float4* a4 = reinterpret_cast<float4*>(P.acc);
    const size_t n4 = (size_t)P.t * P.h / 4;
    for (size_t i = (size_t)blockIdx.x * GV2_THREADS + threadIdx.x; i < n4; i += (size_t)gridDim.x * GV2_THREADS)
      a4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int nkc_all = P.h / GV_KC, nkc = nkc_all / Q.KS;
  const int Iu = blockIdx.y == 1 ? P.Is : P.I;
  const int units_per_e = (Iu / 128) * Q.KS;
  int e, sub;
  bool shared;
  if (!gv2_unit<NB>(P, units_per_e, &s_e, R, e, sub, shared)) return;
  const int rt = sub / Q.KS, ks = sub % Q.KS, kc0 = ks * nkc;
  const int nb = R.n;
  // token rows of this K slice as fp32 (converted once, read by both
  // matrices of every chunk), [NB][nkc * 64]
  float* xs = reinterpret_cast<float*>(ring + GV2_RING);
  float* xch = xs + NB * nkc * GV_KC;  // [128][NB][2] halves exchange
  const int kw = nkc * GV_KC;
  if (threadIdx.x == 0) {
    for (int i = 0; i < ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], GV2_CONS / 32);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort = &abort_flag;
  const uint8_t* rec = shared ? P.s_codes : P.codes + (size_t)e * packed_rec_bytes(P.h, P.I);
  const uint8_t* src = rec + ((size_t)rt * nkc_all + kc0) * 2 * GV_QB;  // [rt][kc][gate][up]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float g[NB], u[NB];
#pragma unroll
  for (int r = 0; r < NB; ++r) g[r] = u[r] = 0.f;
  const int o = threadIdx.x & 127, hf = (threadIdx.x >> 7) & 1;
  // The producer warp starts the weight stream at once; the consumer warps
  // meanwhile stage the token rows (L2 reads) and meet at a named barrier.
  if (warp == GV2_CONS / 32) {
    // no copy under the MOE_STALL_WEIGHT_COPIES test hook: the consumers' waits run out
    // the whole warp walks the loop, one elected lane issues the copies
    if (!(P.status && (P.status->stall & MOE_STALL_WEIGHT_COPIES))) {
      uint32_t armed = 0, par = 0;  // per stage: copy issued, its phase parity (bit masks, not local memory)
      for (int i = 0; i < nkc; ++i) {
        const int s = i % ST;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&empty[s], ((i / ST) & 1) ^ 1, abort, GV2_WAIT_NS))) {
          if (lane == 0) gv2_timeout(P.status, abort, 61);
          break;
        }
        if (elect_one()) {
          mbar_arrive_expect_tx(&full[s], 2 * GV_QB);
          bulk_copy_g2s(ring + s * 2 * GV_QB, src + (size_t)i * 2 * GV_QB, 2 * GV_QB, &full[s]);
        }
        __syncwarp();
        armed |= 1u << s;
        par = (par & ~(1u << s)) | (((i / ST) & 1u) << s);
      }
      if (__any_sync(0xFFFFFFFFu, *abort))
        for (int i = 0; i < ST; ++i)
          if ((armed >> i) & 1u) {
            const int never = 0;
            mbar_wait(&full[i], (par >> i) & 1u, &never, 100000000ull);
          }
    }
  } else {
    for (int v = threadIdx.x; v < nb * kw / 8; v += GV2_CONS) {
      const int r = v / (kw / 8), c = v % (kw / 8);
      const int row = R.row[r];
      uint4 val = make_uint4(0, 0, 0, 0);
      if (row >= 0) val = __ldg(reinterpret_cast<const uint4*>(P.x + (size_t)row * P.h + kc0 * GV_KC) + c);
      float4* d = reinterpret_cast<float4*>(xs + r * kw + c * 8);
      d[0] = make_float4(bf16lo(val.x), bf16hi(val.x), bf16lo(val.y), bf16hi(val.y));
      d[1] = make_float4(bf16lo(val.z), bf16hi(val.z), bf16lo(val.w), bf16hi(val.w));
    }
    asm volatile("bar.sync 1, %0;" ::"n"(GV2_CONS) : "memory");  // consumer warps only
    for (int i = 0; i < nkc; ++i) {
      const int s = i % ST;
      // every lane waits (and so observes the copy); the verdict is made
      // warp-uniform so that a lane giving up cannot leave the others
      // behind at __syncwarp
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[s], (i / ST) & 1, abort, GV2_WAIT_NS))) {
        if (lane == 0) gv2_timeout(P.status, abort, 62);
        break;
      }
      const uint8_t* blk = ring + s * 2 * GV_QB;
      uint32_t wg[16], wu[16];
      dequant_half(blk, o, hf, wg);
      dequant_half(blk + GV_QB, o, hf, wu);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      const float* xk = xs + i * GV_KC + hf * 32;
#pragma unroll
      for (int r = 0; r < NB; ++r)
        if (r < nb) {
          fma32f(wg, xk + r * kw, g[r]);
          fma32f(wu, xk + r * kw, u[r]);
        }
    }
    if (hf == 1)
#pragma unroll
      for (int r = 0; r < NB; ++r)
        if (r < nb) {
          xch[(o * NB + r) * 2] = g[r];
          xch[(o * NB + r) * 2 + 1] = u[r];
        }
  }
  __syncthreads();
  if (threadIdx.x < 128 && !*abort) {
    const int f = rt * 128 + o;
#pragma unroll
    for (int r = 0; r < NB; ++r)
      if (r < nb) {
        float* dst = Q.part + (((size_t)ks * (P.t * P.k + P.t) + R.pos[r]) * 2) * Q.kmax + f;
        dst[0] = g[r] + xch[(o * NB + r) * 2];
        dst[Q.kmax] = u[r] + xch[(o * NB + r) * 2 + 1];
      }
  }
}

// After the last down CTA: out = bf16(acc), or, deterministic mode,
// bf16(acc + sum over the row's list positions in ascending order of
// weight * y) -- the finalize pass, run by the last CTA to finish.
__device__ void gv2_finalize_if_last(const GvParams& P) {
  __shared__ int s_last;
  __shared__ int pos[GV_RB][16];
  __shared__ int npos[GV_RB];
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&P.status->gv_done, 1u) == gridDim.x * gridDim.y - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int r0 = 0; r0 < P.t; r0 += GV_RB) {
    const int nr = min(GV_RB, P.t - r0);
    if (P.deterministic && (int)threadIdx.x < nr) {
      const int r = r0 + threadIdx.x;
      int m = 0;
      for (int j = 0; j < P.k; ++j) {
        const int p = P.slot_of[(size_t)r * P.k + j];
        if (p < 0) continue;
        int i = m++;
        while (i > 0 && pos[threadIdx.x][i - 1] > p) {
          pos[threadIdx.x][i] = pos[threadIdx.x][i - 1];
          --i;
        }
        pos[threadIdx.x][i] = p;
      }
      npos[threadIdx.x] = m;
    }
    __syncthreads();
    for (int v = threadIdx.x; v < nr * P.h / 4; v += blockDim.x) {
      const int rr = v / (P.h / 4), f4 = v % (P.h / 4);
      const int r = r0 + rr;
      float4 a = __ldcg(reinterpret_cast<const float4*>(P.acc + (size_t)r * P.h) + f4);
      if (P.deterministic) {
        for (int j = 0; j < npos[rr]; ++j) {
          const int p = pos[rr][j];
          const float w = P.weights[p];
          const float4 y = __ldcg(reinterpret_cast<const float4*>(P.ybuf + (size_t)p * P.h) + f4);
          a.x = fmaf(w, y.x, a.x);
          a.y = fmaf(w, y.y, a.y);
          a.z = fmaf(w, y.z, a.z);
          a.w = fmaf(w, y.w, a.w);
        }
      }
      uint2 o;
      o.x = pack_bf16x2(a.x, a.y);
      o.y = pack_bf16x2(a.z, a.w);
      reinterpret_cast<uint2*>(P.out + (size_t)r * P.h)[f4] = o;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) P.status->gv_done = 0;
}

// down: unit = (expert, 128-row tile of h).  hg of the unit's rows is
// formed first from the gate/up slices.  Every CTA, with or without a
// unit, counts itself done; the last one finalises the block output.
template <int NB>
__global__ void __launch_bounds__(GV2_THREADS, 1) gv2_down(Gv2Params Q) {
  pdl_wait();
  pdl_trigger();
  const GvParams& P = Q.p;
  extern __shared__ __align__(16) uint8_t sm[];
  uint8_t* ring = sm;
  constexpr int ST = GV2_RING / GV_QB;  // 16 stages of one block
  static_assert(ST <= 32, "stage bit masks");
  __shared__ uint64_t full[ST], empty[ST];
  __shared__ int s_e, abort_flag;
  __shared__ Gv2Rows<NB> R;
  const int Iu = blockIdx.y == 1 ? P.Is : P.I;
  const int units_per_e = P.h / 128;
  int e, rt;
  bool shared;
  if (gv2_unit<NB>(P, units_per_e, &s_e, R, e, rt, shared)) {
    const int nb = R.n, nkc = Iu / GV_KC;
    uint16_t* hs = reinterpret_cast<uint16_t*>(ring + GV2_RING);  // [NB][Iu] bf16
    float* xch = reinterpret_cast<float*>(hs + NB * Iu);
    const size_t pstride = (size_t)(P.t * P.k + P.t) * 2 * Q.kmax;
    if (threadIdx.x == 0) {
      for (int i = 0; i < ST; ++i) {
        mbar_init(&full[i], 1);
        mbar_init(&empty[i], GV2_CONS / 32);
      }
      abort_flag = 0;
      fence_mbar_init();
    }
    __syncthreads();
    volatile int* abort = &abort_flag;
    const uint8_t* rec = shared ? P.s_codes : P.codes + (size_t)e * packed_rec_bytes(P.h, P.I);
    const uint8_t* src = rec + packed_gu_bytes(P.h, Iu) + (size_t)rt * nkc * GV_QB;  // [rt][kc][block]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float y[NB];
#pragma unroll
    for (int r = 0; r < NB; ++r) y[r] = 0.f;
    const int o = threadIdx.x & 127, hf = (threadIdx.x >> 7) & 1;
    // The producer warp starts the weight stream at once; the consumer warps
    // meanwhile form hg from the K-slice partial sums and meet at a named
    // barrier.
    if (warp == GV2_CONS / 32) {
      // no copy under the MOE_STALL_WEIGHT_COPIES test hook: the consumers' waits run out
      // the whole warp walks the loop, one elected lane issues the copies
      if (!(P.status && (P.status->stall & MOE_STALL_WEIGHT_COPIES))) {
        uint32_t armed = 0, par = 0;  // per stage: copy issued, its phase parity (bit masks, not local memory)
        for (int i = 0; i < nkc; ++i) {
          const int s = i % ST;
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(&empty[s], ((i / ST) & 1) ^ 1, abort, GV2_WAIT_NS))) {
            if (lane == 0) gv2_timeout(P.status, abort, 63);
            break;
          }
          if (elect_one()) {
            mbar_arrive_expect_tx(&full[s], GV_QB);
            bulk_copy_g2s(ring + s * GV_QB, src + (size_t)i * GV_QB, GV_QB, &full[s]);
          }
          __syncwarp();
          armed |= 1u << s;
          par = (par & ~(1u << s)) | (((i / ST) & 1u) << s);
        }
        if (__any_sync(0xFFFFFFFFu, *abort))
          for (int i = 0; i < ST; ++i)
            if ((armed >> i) & 1u) {
              const int never = 0;
              mbar_wait(&full[i], (par >> i) & 1u, &never, 100000000ull);
            }
      }
    } else {
      for (int v = threadIdx.x; v < nb * Iu; v += GV2_CONS) {
        const int r = v / Iu, c = v % Iu;
        const float* pp = Q.part + (size_t)R.pos[r] * 2 * Q.kmax + c;
        float gs = 0.f, us = 0.f;
        for (int s = 0; s < Q.KS; ++s) {
          gs += pp[s * pstride];
          us += pp[s * pstride + Q.kmax];
        }
        hs[r * Iu + c] = R.row[r] < 0 ? 0 : f2bf(silu_mul_fast(gs, us));
      }
      asm volatile("bar.sync 1, %0;" ::"n"(GV2_CONS) : "memory");  // consumer warps only
      for (int i = 0; i < nkc; ++i) {
        const int s = i % ST;
        // every lane waits (and so observes the copy); the verdict is made
        // warp-uniform so that a lane giving up cannot leave the others
        // behind at __syncwarp
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[s], (i / ST) & 1, abort, GV2_WAIT_NS))) {
          if (lane == 0) gv2_timeout(P.status, abort, 64);
          break;
        }
        uint32_t wd[16];
        dequant_half(ring + s * GV_QB, o, hf, wd);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        const uint16_t* hk = hs + i * GV_KC + hf * 32;
#pragma unroll
        for (int r = 0; r < NB; ++r)
          if (r < nb) fma32(wd, hk + r * Iu, y[r]);
      }
      if (hf == 1)
#pragma unroll
        for (int r = 0; r < NB; ++r)
          if (r < nb) xch[o * NB + r] = y[r];
    }
    __syncthreads();
    if (threadIdx.x < 128 && !*abort) {
      const int f = rt * 128 + o;
#pragma unroll
      for (int r = 0; r < NB; ++r)
        if (r < nb) {
          const float v = y[r] + xch[o * NB + r];
          const int row = R.row[r];
          if (P.deterministic && !shared) {
            P.ybuf[(size_t)R.pos[r] * P.h + f] = v;
          } else if (row >= 0) {
            float* d = P.acc + (size_t)row * P.h + f;
            if (P.deterministic) *d = R.w[r] * v;
            else atomicAdd(d, R.w[r] * v);
          }
        }
    }
  }
  gv2_finalize_if_last(P);
}

template <int NB>
size_t gv2_smem_gateup(int h, int KS) {
  return GV2_RING + (size_t)NB * (h / KS) * 4 + (size_t)128 * NB * 2 * 4;
}
template <int NB>
size_t gv2_smem_down(int kmax) {
  return GV2_RING + (size_t)NB * kmax * 2 + (size_t)128 * NB * 4;
}

template <int NB>
cudaError_t launch_gv2(const Gv2Params& Q, int nact, cudaStream_t stream) {
  const GvParams& P = Q.p;
  const size_t sg = gv2_smem_gateup<NB>(P.h, Q.KS), sd = gv2_smem_down<NB>(Q.kmax);
  cudaError_t err;
  if ((err = set_smem_limit_once(gv2_gateup<NB>, (int)sg)) != cudaSuccess)
    return err;
  if ((err = set_smem_limit_once(gv2_down<NB>, (int)sd)) != cudaSuccess)
    return err;
  const int ug = (P.I / 128) * Q.KS, ugs = (P.Is / 128) * Q.KS;
  const int xg = nact * ug > ugs ? nact * ug : ugs;
  MOE_LAUNCH("gateup_gemv", stream, (launch_k(gv2_gateup<NB>, dim3(xg, 2), GV2_THREADS, sg, stream, Q)));
  MOE_LAUNCH("down_gemv", stream,
             (launch_k(gv2_down<NB>, dim3(nact * (P.h / 128), 2), GV2_THREADS, sd, stream, Q)));
  return cudaGetLastError();
}

// The streaming variant fits when the staged rows fit next to the ring.
bool gv2_fits(int NB, int h, int kmax, int KS) {
  const size_t lim = 220 * 1024;
  return (size_t)GV2_RING + (size_t)NB * (h / KS) * 4 + (size_t)128 * NB * 8 <= lim &&
         (size_t)GV2_RING + (size_t)NB * kmax * 2 + (size_t)128 * NB * 4 <= lim;
}

template <int NB>
cudaError_t launch_gemv(const GvParams& P, int x_gu, int g_gu, int x_dn, int g_dn, cudaStream_t stream) {
  MOE_LAUNCH("gateup_gemv", stream,
             (launch_k(gemv_kernel<true, NB>, dim3(x_gu, 2), GV_THREADS, 0, stream, P, g_gu)));
  MOE_LAUNCH("down_gemv", stream, (launch_k(gemv_kernel<false, NB>, dim3(x_dn, 2), GV_THREADS, 0, stream, P, g_dn)));
  return cudaGetLastError();
}

}  // namespace

size_t gemv_part_bytes(const moe_dims& d) {
  if (d.t > GV_RB) return 0;
  const size_t kmax = d.inter > d.shared_inter ? d.inter : d.shared_inter;
  return (size_t)GV2_KS_MAX * ((size_t)d.t * d.k + d.t) * 2 * kmax * 4;
}

cudaError_t launch_experts_gemv(const ExpertsArgs& a, bool packed, bool deterministic, cudaStream_t stream) {
  GvParams P{};
  P.t = a.t;
  P.h = a.h;
  P.I = a.I;
  P.Is = a.Is;
  P.E = a.E;
  P.k = a.k;
  P.deterministic = deterministic ? 1 : 0;
  P.packed = packed ? 1 : 0;
  P.x = a.x;
  P.offsets = a.offsets;
  P.rows = a.rows;
  P.weights = a.weights;
  P.codes = a.codes;
  P.scales = a.scales;
  P.biases = a.biases;
  P.s_codes = a.s_codes;
  P.s_scales = a.s_scales;
  P.s_biases = a.s_biases;
  P.hg = a.hg;
  P.hgs = a.hgs;
  P.acc = a.acc;
  P.ybuf = a.ybuf;
  P.status = a.status;
  P.slot_of = a.slot_of;
  P.out = a.out;
  cudaError_t err;
  if (a.Is > 0 && a.s_gate) {
    float* gate_vals = reinterpret_cast<float*>(a.sched);
    if ((err = launch_shared_gate(a.x, a.s_gate, a.t, a.h, gate_vals, stream)) != cudaSuccess) return err;
    P.gate_vals = gate_vals;
  }
  const int nact = a.E < a.t * a.k ? a.E : a.t * a.k;  // experts with a non-empty list, at most
  const int g_gu = a.I / GV_ROWS, g_dn = a.h / GV_ROWS;
  const int gs_gu = a.Is / GV_ROWS;
  const int x_gu = nact * g_gu > gs_gu ? nact * g_gu : gs_gu;
  const int rows = a.t < GV_RB ? a.t : GV_RB;
  const int NBr = rows <= 1 ? 1 : rows <= 2 ? 2 : rows <= 4 ? 4 : rows <= 8 ? 8 : 16;
  const int kmax = a.I > a.Is ? a.I : a.Is;
  if (packed && a.t <= GV_RB && a.gvpart) {
    // K slices: enough units to occupy the GPU when few experts are active
    // (measured: 8 slices at 48 gate/up units beat 2; at 96 units one slice
    // beats four, the per-CTA fixed cost outweighing the better spread)
    const int units = nact * (a.I / 128);
    const int nkc = a.h / GV_KC;
    int KS = units < 60 ? 8 : units < 80 ? 2 : 1;
    while (KS > 1 && (nkc % KS || !gv2_fits(NBr, a.h, kmax, KS))) KS >>= 1;
    if (gv2_fits(NBr, a.h, kmax, KS)) {
      Gv2Params Q{P, a.gvpart, KS, kmax};
      if (NBr == 1) err = launch_gv2<1>(Q, nact, stream);
      else if (NBr == 2) err = launch_gv2<2>(Q, nact, stream);
      else if (NBr == 4) err = launch_gv2<4>(Q, nact, stream);
      else if (NBr == 8) err = launch_gv2<8>(Q, nact, stream);
      else err = launch_gv2<16>(Q, nact, stream);
      return err;  // gv2_down's last CTA has written out
    }
  }
  if (rows <= 1) err = launch_gemv<1>(P, x_gu, g_gu, nact * g_dn, g_dn, stream);
  else if (rows <= 2) err = launch_gemv<2>(P, x_gu, g_gu, nact * g_dn, g_dn, stream);
  else if (rows <= 4) err = launch_gemv<4>(P, x_gu, g_gu, nact * g_dn, g_dn, stream);
  else if (rows <= 8) err = launch_gemv<8>(P, x_gu, g_gu, nact * g_dn, g_dn, stream);
  else err = launch_gemv<16>(P, x_gu, g_gu, nact * g_dn, g_dn, stream);
  if (err != cudaSuccess) return err;
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  return launch_finalize(a, deterministic, stream);
}

}  // namespace moe

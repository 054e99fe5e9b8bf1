// Router on the tensor cores, exact in the canonical fp32 order
// (cherenkov qwen4_exp, prefill.rs, pf_layer -> router_b: logits = x Wr^T,
// top-k, softmax over the selected logits).
//
// Two kernels:
//   route_score:  approximate scores S = x Wr^T with tcgen05 (bf16 operands
//     staged by TMA, fp32 accumulator in TMEM) over tiles of 128 rows x NT
//     experts, with the K range split into KS slices whose partial sums are
//     stored side by side (no atomics).  While the MMAs run, the four
//     epilogue warps compute the squared norms |w_e|^2 of the router rows.
//   route_refine: one warp per row, or two for short chunks (they split the
//     recomputations, so that a few hundred rows still fill the GPU).  The score a_e (slices summed, bias
//     added) differs from the canonical fp32 logit c_e by at most
//       D_e = eps * |x| * |w_e| + 2^-21 |a_e|,
//     because sum_i |x_i w_ei| <= |x| |w_e| (Cauchy-Schwarz) and eps covers
//     the tensor core's fp32 accumulation, the canonical order's own
//     rounding and the slice sums with a wide margin.  With L the k-th
//     largest of a_e - D_e, every expert with a_e + D_e >= L is a
//     candidate: k experts have c >= L, so an expert below that cannot be
//     in the top-k.  The candidates' logits are recomputed in the canonical
//     order, and the selection and softmax run on those exact values, so
//     idx and w are bit-identical to the single-pass exact kernel's.
//     Rows with a non-finite norm or score take every expert as candidate.
//     Each recomputed candidate also checks |a_e - c_e| <= D_e; the largest
//     ratio is kept in the workspace status block and a violation raises
//     FLAG_ROUTE_BOUND.
#include "route_common.cuh"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int RS_STAGES = 4;
constexpr int RS_WARPS = 6;  // 0 TMA producer, 1 MMA issuer (+ TMEM), 2-5 epilogue
constexpr int RS_KC = 64;    // K per stage: one 128-byte swizzled row
constexpr int RS_A_BYTES = 128 * 128;
constexpr uint64_t RS_WAIT_NS = 2000000000ull;
constexpr int RS_TARGET_CTAS = 152;  // about one CTA per SM of a GB300
constexpr int RS_KS_MAX = 4;         // K slices: each costs the refinement one more load per score
constexpr int RF_WARPS = 8;  // 4 rows per CTA, two warps each
constexpr int RF_NB = 2;  // exact logits computed together per warp (4 measured slower: fewer batches, but spills)

struct ScoreParams {
  int t, h, E, Ep, NT, nkc_split;
  float* part;  // [KS][t][Ep] partial scores
  float* wn2;   // [E] squared router-row norms
  const uint16_t* wr;
  DeviceStatus* st;
};

__device__ __forceinline__ void rs_timeout(DeviceStatus* st, volatile int* abort, uint32_t site) {
  if (atomicOr(&st->flags, FLAG_TIMEOUT) == 0) st->timeout_site = site;
  *abort = 1;
}

__device__ __forceinline__ void rs_drain_wait(uint64_t* bar, uint32_t parity) {
  const int never = 0;
  mbar_wait(bar, parity, &never, 100000000ull);
}

__device__ __forceinline__ float sumsq8(uint4 u) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = bf16lo(w[i]), b = bf16hi(w[i]);
    s = fmaf(a, a, s);
    s = fmaf(b, b, s);
  }
  return s;
}

__global__ void __launch_bounds__(RS_WARPS * 32, 1)
route_score_kernel(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap tw, ScoreParams P) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[RS_STAGES], empty[RS_STAGES], accf, drain;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int NT = P.NT;
  const uint32_t st_bytes = RS_A_BYTES + NT * 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.x * 128, e0 = blockIdx.y * NT, ks = blockIdx.z;
  const int kc0 = ks * P.nkc_split;
  const int nkc = min(P.nkc_split, P.h / RS_KC - kc0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < RS_STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(&accf, 1);
    mbar_init(&drain, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&tmem_slot, NT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort = &abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tx);
      prefetch_tmap(&tw);
      uint32_t armed = 0, par = 0;  // per stage: copy issued, its phase parity (bit masks, not local memory)
      for (int i = 0; i < nkc; ++i) {
        const int s = i % RS_STAGES;
        if (!mbar_wait(&empty[s], ((i / RS_STAGES) & 1) ^ 1, abort, RS_WAIT_NS)) {
          rs_timeout(P.st, abort, 51);
          break;
        }
        uint8_t* sa = base + s * st_bytes;
        mbar_arrive_expect_tx(&full[s], st_bytes);
        tma_load_2d(sa, &tx, (kc0 + i) * RS_KC, row0, &full[s]);
        tma_load_2d(sa + RS_A_BYTES, &tw, (kc0 + i) * RS_KC, e0, &full[s]);
        armed |= 1u << s;
        par = (par & ~(1u << s)) | (((i / RS_STAGES) & 1u) << s);
      }
      if (*abort)
        for (int i = 0; i < RS_STAGES; ++i)
          if ((armed >> i) & 1u) rs_drain_wait(&full[i], (par >> i) & 1u);
    }
  } else if (warp == 1) {
    // MMA issuer: the whole warp walks the loop, one elected lane (the same
    // one every time, so the commits track its MMAs) issues
    const uint32_t idesc = idesc_bf16(128, NT);
    bool ok = true;
    for (int i = 0; i < nkc; ++i) {
      const int s = i % RS_STAGES;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[s], (i / RS_STAGES) & 1, abort, RS_WAIT_NS))) {
        if (lane == 0) rs_timeout(P.st, abort, 52);
        ok = false;
        break;
      }
      if (elect_one()) {
        tc_fence_after();
        const uint32_t sa = smem_u32(base + s * st_bytes);
        const uint64_t ad = desc_sw128(sa), bd = desc_sw128(sa + RS_A_BYTES);
#pragma unroll
        for (int kk = 0; kk < RS_KC / 16; ++kk) mma_bf16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (i | kk) != 0);
        mma_commit(&empty[s]);
      }
      __syncwarp();
    }
    if (elect_one()) mma_commit(ok ? &accf : &drain);
    __syncwarp();
    if (!ok) rs_drain_wait(&drain, 0);
  } else {
    // Squared norms of this column's router rows, spread over the CTAs that
    // share the column (rows r = 4 * li + ew, stepping by 4 * nl).
    const int ew = warp - 2, q = warp & 3;
    const int nl = gridDim.x * gridDim.z, li = blockIdx.z * gridDim.x + blockIdx.x;
    for (int r = li * 4 + ew; r < NT && e0 + r < P.E; r += nl * 4) {
      const uint4* wrow = reinterpret_cast<const uint4*>(P.wr + (size_t)(e0 + r) * P.h);
      float s2 = 0.f;
      for (int v = lane; v < P.h / 8; v += 32) s2 += sumsq8(__ldg(wrow + v));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s2 += __shfl_xor_sync(0xFFFFFFFFu, s2, o);
      if (lane == 0) P.wn2[e0 + r] = s2;
    }
    // warp-uniform verdict: tcgen05.ld below is .sync.aligned
    if (__all_sync(0xFFFFFFFFu, mbar_wait(&accf, 0, abort, RS_WAIT_NS))) {
      tc_fence_after();
      const int row = row0 + q * 32 + lane;
      float* dst = P.part + ((size_t)ks * P.t + row) * P.Ep + e0;
      for (int c = 0; c < NT / 16; ++c) {
        uint32_t y[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + c * 16, y);
        tmem_ld_wait();
        tmem_ld_fence(y);
        if (row < P.t && e0 + c * 16 < P.Ep) {
          float4* d4 = reinterpret_cast<float4*>(dst + c * 16);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            d4[j] = make_float4(__uint_as_float(y[4 * j]), __uint_as_float(y[4 * j + 1]),
                                __uint_as_float(y[4 * j + 2]), __uint_as_float(y[4 * j + 3]));
        }
      }
    } else if (lane == 0 && !*abort) {
      rs_timeout(P.st, abort, 53);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, NT);
  }
}

// Canonical-order logits of NB (row, expert) pairs of one row: for each,
// lane l sums the exact bf16 products of K = 256 m + 8 l + c from +0, m then
// c ascending (zeros past h), and the lane sums combine by the xor butterfly
// 16, 8, 4, 2, 1, so every lane ends with the same value.  The NB chains are
// independent and interleaved, each in its own order.
template <int NB>
__device__ __forceinline__ void canonical_dots(const uint16_t* xr, const uint16_t* const (&wrow)[NB], int h, int nm,
                                               int lane, float (&P)[NB]) {
#pragma unroll
  for (int j = 0; j < NB; ++j) P[j] = 0.f;
  int m = 0;
  for (; m + 4 <= nm; m += 4) {
    uint4 xv[4], wv[4][NB];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int k0 = (m + u) * 256 + lane * 8;
      const bool in = k0 < h;
      xv[u] = in ? __ldg(reinterpret_cast<const uint4*>(xr + k0)) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int j = 0; j < NB; ++j)
        wv[u][j] = in ? __ldg(reinterpret_cast<const uint4*>(wrow[j] + k0)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t xw = (&xv[u].x)[c >> 1];
        const float xf = (c & 1) ? bf16hi(xw) : bf16lo(xw);
#pragma unroll
        for (int j = 0; j < NB; ++j) {
          const uint32_t ww = (&wv[u][j].x)[c >> 1];
          P[j] = fmaf(xf, (c & 1) ? bf16hi(ww) : bf16lo(ww), P[j]);
        }
      }
  }
  for (; m < nm; ++m) {
    const int k0 = m * 256 + lane * 8;
    const bool in = k0 < h;
    const uint4 xv = in ? __ldg(reinterpret_cast<const uint4*>(xr + k0)) : make_uint4(0, 0, 0, 0);
    uint4 wv[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j)
      wv[j] = in ? __ldg(reinterpret_cast<const uint4*>(wrow[j] + k0)) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint32_t xw = (&xv.x)[c >> 1];
      const float xf = (c & 1) ? bf16hi(xw) : bf16lo(xw);
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        const uint32_t ww = (&wv[j].x)[c >> 1];
        P[j] = fmaf(xf, (c & 1) ? bf16hi(ww) : bf16lo(ww), P[j]);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int j = 0; j < NB; ++j) P[j] = P[j] + __shfl_xor_sync(0xFFFFFFFFu, P[j], o);
}

template <int NQ, int WPR>  // WPR warps per row (1 or 2)
__global__ void __launch_bounds__(RF_WARPS * 32, 4)
route_refine_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr, const float* __restrict__ rbias,
                    const float* __restrict__ part, int KS, int Ep, const float* __restrict__ wn2, int t, int h,
                    int E, int k, float eps, int32_t* __restrict__ idx, float* __restrict__ wout,
                    DeviceStatus* st) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int pair = warp / WPR, half = warp % WPR;  // the warps of a row
  const int row = blockIdx.x * (RF_WARPS / WPR) + pair;
  if (row >= t) return;  // the warps of a row leave together
  const int nm = (h + 255) / 256;
  const uint16_t* xr = x + (size_t)row * h;

  float xs2 = 0.f;
#pragma unroll 4
  for (int m = 0; m < nm; ++m) {
    const int k0 = m * 256 + lane * 8;
    if (k0 < h) xs2 += sumsq8(__ldg(reinterpret_cast<const uint4*>(xr + k0)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) xs2 += __shfl_xor_sync(0xFFFFFFFFu, xs2, o);
  const float xn = sqrtf(xs2);

  float av[NQ], dv[NQ];
  bool finite = isfinite(xn);
  // slice sums (any order: the bound allows for it), all loads of a slice in flight together
#pragma unroll
  for (int q = 0; q < NQ; ++q) av[q] = 0.f;
#pragma unroll 4
  for (int s = 0; s < KS; ++s) {
    const float* ps = part + ((size_t)s * t + row) * Ep + lane;
#pragma unroll
    for (int q = 0; q < NQ; ++q)
      if (lane + 32 * q < E) av[q] += __ldg(ps + 32 * q);
  }
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    const int e = lane + 32 * q;
    const float a0 = av[q];
    av[q] = -INFINITY;
    dv[q] = 0.f;
    if (e < E) {
      float a = a0;
      if (rbias) a += rbias[e];
      const float d = eps * xn * sqrtf(wn2[e]) + 0x1p-21f * fabsf(a) + 1e-30f;
      av[q] = a;
      dv[q] = d;
      finite = finite && isfinite(a) && isfinite(d);
    }
  }
  finite = __all_sync(0xFFFFFFFFu, finite);

  // L = k-th largest lower bound (with multiplicity).
  float L = -INFINITY;
  if (finite) {
    uint32_t removed = 0;
    for (int j = 0; j < k; ++j) {
      float best = -INFINITY;
      int bq = -1;
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        const float lb = av[q] - dv[q];
        if (lane + 32 * q < E && !((removed >> q) & 1u) && (bq < 0 || lb > best)) best = lb, bq = q;
      }
      float wbest = best;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) wbest = fmaxf(wbest, __shfl_xor_sync(0xFFFFFFFFu, wbest, o));
      const uint32_t who = __ballot_sync(0xFFFFFFFFu, bq >= 0 && best == wbest);
      if (lane == __ffs(who) - 1) removed |= 1u << bq;
      L = wbest;
    }
  }

  // Candidate list of this row, then exact logits in batches of RF_NB.
  // per pair: the second warp's keys [NQ * 32] and the candidate list [NQ * 32]
  extern __shared__ __align__(16) unsigned char rf_smem[];
  uint64_t* key_s = reinterpret_cast<uint64_t*>(rf_smem) + (size_t)pair * NQ * 32;
  int* cl = reinterpret_cast<int*>(reinterpret_cast<uint64_t*>(rf_smem) + (size_t)(RF_WARPS / WPR) * NQ * 32) +
            (size_t)pair * NQ * 32;
  __shared__ float audit_s[RF_WARPS];
  int ncand = 0;
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    const bool cand = (lane + 32 * q < E) && (!finite || av[q] + dv[q] >= L);
    const uint32_t mask = __ballot_sync(0xFFFFFFFFu, cand);
    if (cand && half == 0) cl[ncand + __popc(mask & ((1u << lane) - 1u))] = lane + 32 * q;
    ncand += __popc(mask);
  }
  if (WPR == 2) asm volatile("bar.sync %0, 64;" ::"r"(1 + pair) : "memory");  // the list is complete for both warps
  else __syncwarp();
  uint64_t key[NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) key[q] = 0ull;
  float audit = 0.f;
  // the pair's warps take alternate batches of RF_NB candidates
  for (int b = half * RF_NB; b < ncand; b += WPR * RF_NB) {
    int e[RF_NB];
    const uint16_t* wrow[RF_NB];
#pragma unroll
    for (int j = 0; j < RF_NB; ++j) {
      e[j] = cl[min(b + j, ncand - 1)];
      wrow[j] = wr + (size_t)e[j] * h;
    }
    float c[RF_NB];
    canonical_dots<RF_NB>(xr, wrow, h, nm, lane, c);
#pragma unroll
    for (int j = 0; j < RF_NB; ++j) {
      if (b + j < ncand && lane == (e[j] & 31)) {
        const float cj = rbias ? c[j] + rbias[e[j]] : c[j];
#pragma unroll
        for (int q = 0; q < NQ; ++q)
          if (q == (e[j] >> 5)) {
            key[q] = topk_key(cj, e[j]);
            if (finite) audit = fmaxf(audit, fabsf(av[q] - cj) / dv[q]);
          }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) audit = fmaxf(audit, __shfl_xor_sync(0xFFFFFFFFu, audit, o));
  if (WPR == 2) {
    // merge the second warp's keys (each expert's key is set by exactly one warp)
    if (half == 1) {
#pragma unroll
      for (int q = 0; q < NQ; ++q) key_s[q * 32 + lane] = key[q];
      if (lane == 0) audit_s[pair] = audit;
    }
    asm volatile("bar.sync %0, 64;" ::"r"(1 + pair) : "memory");
    if (half == 1) return;
#pragma unroll
    for (int q = 0; q < NQ; ++q) key[q] |= key_s[q * 32 + lane];
    audit = fmaxf(audit, audit_s[pair]);
  }
  if (lane == 0) {
    if (audit > 0.f) atomicMax(&st->route_audit, __float_as_uint(audit));
    atomicAdd(&st->route_cands, (uint32_t)ncand);
    if (!(audit <= 1.f)) raise_flag(st, FLAG_ROUTE_BOUND);
  }
  warp_topk_softmax<NQ>(key, k, lane, idx + (size_t)row * k, wout + (size_t)row * k);
}

// Small t (at most RSM_ROWS rows): every logit in the canonical order, one
// warp per expert over all rows (the router row is read once, RSM_UNROLL
// K spans of it in flight per lane), then the last CTA to finish selects
// the top-k of every row.
constexpr int RSM_ROWS = 16;
constexpr int RSM_WARPS = 4;

// The grouping of moe_build_csr for at most 256 pairs (t <= 16, k <= 16),
// by the router's last block once every row's top k is written: per-expert
// counts in shared memory, one scan over the experts (eight per thread), and
// each pair's rank inside its expert by counting the earlier pairs of the same
// expert -- the same stable order as the grouping kernels.
__device__ __forceinline__ void small_csr_block(const int32_t* idx, const float* w, int n, int k, int E,
                                                const moe_csr& co, DeviceStatus* st) {
  constexpr int T = RSM_WARPS * 32, PER = 1024 / T;
  __shared__ int start[1024];
  __shared__ int es[256];
  __shared__ int warp_sums[RSM_WARPS + 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < E; i += T) start[i] = 0;
  for (int p = tid; p < n; p += T) {
    int e = __ldcg(idx + p);  // written by this block before the barrier
    if (e < 0 || e >= E) {
      raise_flag(st, FLAG_BAD_EXPERT);
      e = -1;
    }
    es[p] = e;
  }
  __syncthreads();
  for (int p = tid; p < n; p += T)
    if (es[p] >= 0) atomicAdd(&start[es[p]], 1);
  __syncthreads();
  int c[PER], sum = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int ex = tid * PER + j;
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
  if (tid == 0) {
    int run = 0;
    for (int i = 0; i < RSM_WARPS; ++i) {
      const int v = warp_sums[i];
      warp_sums[i] = run;
      run += v;
    }
    warp_sums[RSM_WARPS] = run;
  }
  __syncthreads();
  int run = warp_sums[warp] + incl - sum;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int ex = tid * PER + j;
    if (ex < E) {
      start[ex] = run;
      co.offsets[ex] = run;
    }
    run += c[j];
  }
  if (tid == 0) co.offsets[E] = warp_sums[RSM_WARPS];
  __syncthreads();
  for (int p = tid; p < n; p += T) {
    const int e = es[p];
    if (e < 0) {
      co.slot_of[p] = -1;
      continue;
    }
    int r = 0;
    for (int q = 0; q < p; ++q) r += es[q] == e;
    const int pos = start[e] + r;
    co.rows[pos] = p / k;
    co.weights[pos] = __ldcg(w + p);
    co.slot_of[p] = pos;
  }
}

template <int TR, int NQ>
__global__ void __launch_bounds__(RSM_WARPS * 32)
route_small_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr, const float* __restrict__ rbias,
                   int t, int h, int E, int Ep, int k, float* lg, int32_t* __restrict__ idx, float* __restrict__ wout,
                   DeviceStatus* st, moe_csr co) {
  pdl_wait();
  pdl_trigger();
  constexpr int U = TR <= 2 ? 8 : (TR <= 4 ? 4 : 2);  // K spans per load round
  __shared__ int is_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e = blockIdx.x * RSM_WARPS + warp;
  const int nm = (h + 255) / 256;
  if (e < E) {
    float P[TR];
#pragma unroll
    for (int r = 0; r < TR; ++r) P[r] = 0.f;
    const uint16_t* wrow = wr + (size_t)e * h;
    for (int m0 = 0; m0 < nm; m0 += U) {
      uint4 wv[U], xv[U][TR];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int k0 = (m0 + u) * 256 + lane * 8;
        const bool in = m0 + u < nm && k0 < h;
        wv[u] = in ? __ldg(reinterpret_cast<const uint4*>(wrow + k0)) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int r = 0; r < TR; ++r)
          xv[u][r] = (in && r < t) ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)r * h + k0))
                                   : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (m0 + u >= nm) break;  // spans past the padded width add nothing
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t ww = (&wv[u].x)[c >> 1];
          const float wf = (c & 1) ? bf16hi(ww) : bf16lo(ww);
#pragma unroll
          for (int r = 0; r < TR; ++r) {
            const uint32_t xw = (&xv[u][r].x)[c >> 1];
            P[r] = fmaf((c & 1) ? bf16hi(xw) : bf16lo(xw), wf, P[r]);
          }
        }
      }
    }
    const float b = rbias ? rbias[e] : 0.f;
#pragma unroll
    for (int r = 0; r < TR; ++r) {
      float v = P[r];
      v = v + __shfl_xor_sync(0xFFFFFFFFu, v, 16);
      v = v + __shfl_xor_sync(0xFFFFFFFFu, v, 8);
      v = v + __shfl_xor_sync(0xFFFFFFFFu, v, 4);
      v = v + __shfl_xor_sync(0xFFFFFFFFu, v, 2);
      v = v + __shfl_xor_sync(0xFFFFFFFFu, v, 1);
      if (lane == r && r < t) lg[(size_t)r * Ep + e] = rbias ? v + b : v;
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(&st->route_done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  for (int r = warp; r < t; r += RSM_WARPS) {
    uint64_t key[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const int ee = lane + 32 * q;
      key[q] = ee < E ? topk_key(__ldcg(lg + (size_t)r * Ep + ee), ee) : 0ull;
    }
    warp_topk_softmax<NQ>(key, k, lane, idx + (size_t)r * k, wout + (size_t)r * k);
  }
  if (co.offsets) {
    __syncthreads();  // every row's idx and w are written
    small_csr_block(idx, wout, t * k, k, E, co, st);
  }
  if (threadIdx.x == 0) st->route_done = 0;
}

struct RoutePlan {
  int Ep, NT, mt, ntn, nk, KS, nkc_split;
};

RoutePlan route_plan(int t, int h, int E) {
  RoutePlan R;
  R.Ep = (E + 15) / 16 * 16;
  R.NT = 32;
  while (R.NT < E && R.NT < 256) R.NT *= 2;
  R.mt = (t + 127) / 128;
  R.ntn = (E + R.NT - 1) / R.NT;
  R.nk = h / RS_KC;
  int ks = RS_TARGET_CTAS / (R.mt * R.ntn);
  ks = ks < R.nk / 2 ? ks : R.nk / 2;
  ks = ks < RS_KS_MAX ? ks : RS_KS_MAX;
  if (ks < 1) ks = 1;
  R.nkc_split = (R.nk + ks - 1) / ks;
  R.KS = (R.nk + R.nkc_split - 1) / R.nkc_split;
  return R;
}

size_t score_smem_bytes(int NT) { return 1024 + (size_t)RS_STAGES * (RS_A_BYTES + NT * 128); }

template <int NQ, int WPR>
cudaError_t launch_refine_w(const uint16_t* x, const uint16_t* wr, const float* rbias, const float* part,
                            const RoutePlan& R, const float* wn2, int t, int h, int E, int k, float eps, int32_t* idx,
                            float* w, DeviceStatus* st, cudaStream_t stream) {
  const size_t smem = (size_t)(RF_WARPS / WPR) * NQ * 32 * 12;
  const cudaError_t e = set_smem_limit_once(route_refine_kernel<NQ, WPR>, (int)smem);
  if (e != cudaSuccess) return e;
  const int rows_per_cta = RF_WARPS / WPR;
  MOE_LAUNCH("route_refine", stream,
             (launch_k(route_refine_kernel<NQ, WPR>, (t + rows_per_cta - 1) / rows_per_cta, RF_WARPS * 32, smem, stream, 
                 x, wr, rbias, part, R.KS, R.Ep, wn2, t, h, E, k, eps, idx, w, st)));
  return cudaGetLastError();
}

// Two warps per row while one warp per row would leave most SMs idle.
template <int NQ>
cudaError_t launch_refine(const uint16_t* x, const uint16_t* wr, const float* rbias, const float* part,
                          const RoutePlan& R, const float* wn2, int t, int h, int E, int k, float eps, int32_t* idx,
                          float* w, DeviceStatus* st, cudaStream_t stream) {
  if (t <= 1024) return launch_refine_w<NQ, 2>(x, wr, rbias, part, R, wn2, t, h, E, k, eps, idx, w, st, stream);
  return launch_refine_w<NQ, 1>(x, wr, rbias, part, R, wn2, t, h, E, k, eps, idx, w, st, stream);
}

template <int TR, int NQ>
cudaError_t launch_small_t(const uint16_t* x, const uint16_t* wr, const float* rbias, int t, int h, int E, int k,
                           float* lg, int32_t* idx, float* w, DeviceStatus* st, const moe_csr* co,
                           cudaStream_t stream) {
  MOE_LAUNCH("route_small", stream,
             launch_k(route_small_kernel<TR, NQ>, (E + RSM_WARPS - 1) / RSM_WARPS, RSM_WARPS * 32, 0, stream, 
                 x, wr, rbias, t, h, E, (E + 15) / 16 * 16, k, lg, idx, w, st, co ? *co : moe_csr{}));
  return cudaGetLastError();
}

template <int NQ>
cudaError_t launch_small(const uint16_t* x, const uint16_t* wr, const float* rbias, int t, int h, int E, int k,
                         float* lg, int32_t* idx, float* w, DeviceStatus* st, const moe_csr* co,
                         cudaStream_t stream) {
  if (t <= 1) return launch_small_t<1, NQ>(x, wr, rbias, t, h, E, k, lg, idx, w, st, co, stream);
  if (t <= 2) return launch_small_t<2, NQ>(x, wr, rbias, t, h, E, k, lg, idx, w, st, co, stream);
  if (t <= 4) return launch_small_t<4, NQ>(x, wr, rbias, t, h, E, k, lg, idx, w, st, co, stream);
  if (t <= 8) return launch_small_t<8, NQ>(x, wr, rbias, t, h, E, k, lg, idx, w, st, co, stream);
  return launch_small_t<16, NQ>(x, wr, rbias, t, h, E, k, lg, idx, w, st, co, stream);
}

}  // namespace

size_t route_ws_bytes(int t, int h, int E) {
  const RoutePlan R = route_plan(t, h, E);
  return align_up((size_t)R.KS * t * R.Ep * 4, 256) + align_up((size_t)E * 4, 256);
}


// Whether launch_route_tc builds the grouping itself when given one (the
// small-t router's last block does, for t <= 16 rows).
bool route_builds_csr(int t) { return t <= RSM_ROWS; }

cudaError_t launch_route_tc(const uint16_t* x, const uint16_t* wr, const float* rbias, int t, int h, int E, int k,
                            int32_t* idx, float* w, unsigned char* scratch, DeviceStatus* st, cudaStream_t stream,
                            const moe_csr* co) {
  const RoutePlan R = route_plan(t, h, E);
  float* part = reinterpret_cast<float*>(scratch);
  if (t <= RSM_ROWS) {
    if (E <= 128) return launch_small<4>(x, wr, rbias, t, h, E, k, part, idx, w, st, co, stream);
    if (E <= 256) return launch_small<8>(x, wr, rbias, t, h, E, k, part, idx, w, st, co, stream);
    if (E <= 512) return launch_small<16>(x, wr, rbias, t, h, E, k, part, idx, w, st, co, stream);
    return launch_small<32>(x, wr, rbias, t, h, E, k, part, idx, w, st, co, stream);
  }
  float* wn2 = reinterpret_cast<float*>(scratch + align_up((size_t)R.KS * t * R.Ep * 4, 256));
  CUtensorMap tx, tw;
  cudaError_t err;
  if ((err = tmap_2d(&tx, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h, t, (uint64_t)h * 2, RS_KC, 128,
                     CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return err;
  if ((err = tmap_2d(&tw, wr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h, E, (uint64_t)h * 2, RS_KC, R.NT,
                     CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return err;
  const size_t smem = score_smem_bytes(R.NT);
  if ((err = set_smem_limit_once(route_score_kernel, (int)score_smem_bytes(256))) != cudaSuccess) return err;
  ScoreParams P{t, h, E, R.Ep, R.NT, R.nkc_split, part, wn2, wr, st};
  MOE_LAUNCH("route_score", stream,
             launch_k(route_score_kernel, dim3(R.mt, R.ntn, R.KS), RS_WARPS * 32, smem, stream, tx, tw, P));
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  // eps: tensor-core accumulation (h 2^-21), canonical order and slice sums
  // ((h/32 + 8 + KS) 2^-23), norm rounding (factor 1 + h 2^-22).
  const double eps = ((double)h * 0x1p-21 + ((double)h / 32 + 8 + R.KS) * 0x1p-23) * (1.0 + (double)h * 0x1p-22);
  const float fe = (float)eps;
  if (E <= 128) return launch_refine<4>(x, wr, rbias, part, R, wn2, t, h, E, k, fe, idx, w, st, stream);
  if (E <= 256) return launch_refine<8>(x, wr, rbias, part, R, wn2, t, h, E, k, fe, idx, w, st, stream);
  if (E <= 512) return launch_refine<16>(x, wr, rbias, part, R, wn2, t, h, E, k, fe, idx, w, st, stream);
  return launch_refine<32>(x, wr, rbias, part, R, wn2, t, h, E, k, fe, idx, w, st, stream);
}

}  // namespace moe

// The whole routed-MoE block for a decode-shaped chunk (t <= 8 rows) in one
// persistent launch: the router (cherenkov qwen4_exp, prefill.rs, pf_layer ->
// router_b), the grouping (prefill/experts.rs, prepare_expert_jobs) and the
// expert FFNs (prefill/experts.rs, pf_experts: gate/up quantised matmuls ->
// silu_mul -> down quantised matmul -> weighted scatter-add, plus the shared
// expert): the MoE part of the multi-row step that decode.rs, step_rows,
// runs per verify batch.
//
// At this size the work is bound by the expert weight bytes (each byte is
// used by at most t dot products) and by latency: a chain of separate
// launches pays each kernel's ramp-up and its own round trips to memory.
// One cooperative grid of one CTA per SM replaces the kernel boundaries with
// counters in the workspace.
//
// Work: the gate/up block pairs and the down blocks of the shared expert and
// of every touched expert, split evenly over the CTAs, each CTA taking one
// contiguous range of each, in the order
//   A. its share of the shared expert's gate/up pairs (known before routing),
//   B. its share of the touched experts' gate/up pairs,
//   C. its share of the shared expert's down blocks,
//   D. its share of the touched experts' down blocks.
//
// Warp roles (14 warps):
//   0      producer: one thread bulk-copies the blocks of the CTA's items
//          into a ring in shared memory, starting with part A at once;
//   1      MMA issuer: one thread issues tcgen05.mma (M = 128 weight rows,
//          N = 16 token columns, A in tensor memory, B in shared memory);
//   2-9    two dequantisation groups taking alternate items: one weight row
//          per thread, w = fma(q, s, b) in bf16 (one rounding) straight into
//          tensor memory (tcgen05.st);
//   10-13  first the router: the logits of experts b, b + G, ... in the
//          fixed summation order of moe_route_topk (lane l owns
//          K = 256 m + 8 l + c, m then c ascending from +0, lane sums
//          combined by the xor butterfly 16..1, bias last), zeroing of the
//          accumulators, a grid-wide barrier (a generation counter every call
//          advances by the grid size), top-k and grouping (identical in every
//          CTA; CTA 0 writes idx, w and the CSR arrays); then the epilogue:
//          tcgen05.ld of the accumulators and fp32 atomics into the
//          per-expert gate/up sums and into the block accumulator.
//
// Operands.  Gate/up: B is x, staged once as 64-wide K chunks of 16 rows
// (128-byte swizzled, rows past t zero), so every expert is multiplied with
// all t rows -- at N = 16 the MMA costs the same -- and the epilogue keeps
// the columns of the expert's own rows.  Down: B is silu(gate) * up of one
// 64-wide chunk for the expert's rows (rounded to bf16, as the hidden
// activations are everywhere else), built by the epilogue warps once the
// chunk's gate/up sums are complete: a counter per (expert, 128-row feature
// tile) counts the K chunks added.  A counter per 128-column output tile lets
// the last contributor round the tile to bf16.
//
// Every wait is bounded (2 s of global time): a wait that gives up records
// MOE_ETIMEOUT, the CTA stops, lets its in-flight copies and MMAs land, frees
// its tensor memory and returns.  moe_read_device_status() then clears the
// counters, so the next call starts clean.
#include "experts.cuh"
#include "route_common.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int D_WARPS = 14;
constexpr int D_THREADS = D_WARPS * 32;
constexpr int W_PROD = 0, W_ISSUE = 1, W_DQ0 = 2, W_EPI0 = 10;
constexpr int D_SLOT = 2 * PACK_QB;  // ring slot: a gate/up block pair (a down block uses half)
constexpr int D_NSLOT = 12;
constexpr int D_NA = 4;              // tensor-memory A slots of 64 columns (a gate/up pair, or a down block)
constexpr int D_NACC = 8;            // accumulator buffers of 32 columns (gate 16 + up 16, or down 16)
constexpr int D_ACC_COL = D_NA * 64;
constexpr int D_NHG = 4;             // silu(gate) * up tiles of the down pass
constexpr int D_TILE = 2048;         // 16 rows x 128 bytes, swizzled
constexpr int D_MAX_H = 2048;        // x is staged as h / 64 tiles
constexpr int D_MAX_T = 8;
constexpr int D_MAX_E = 256;
constexpr int D_MAX_PAIRS = D_MAX_T * 16;
constexpr int D_KC = 64;
constexpr uint64_t D_WAIT_NS = 2000000000ull;

struct DfParams {
  int t, h, I, Is, E, Ep, k;
  const uint16_t* x;        // bf16 [t][h]
  const uint16_t* wr;       // bf16 [E][h]
  const float* rbias;       // [E] or null
  const uint16_t* s_gate;   // bf16 [h] or null
  const uint8_t* packed;    // routed records (moe_pack_experts)
  const uint8_t* s_packed;  // shared record (Is > 0)
  int32_t* idx;             // [t][k] out
  float* w;                 // [t][k] out
  moe_csr csr;              // out
  uint16_t* out;            // bf16 [t][h] out
  float* logits;            // ws: [t][Ep]
  float* gate_vals;         // ws: [t]
  float* gu;                // ws: [slots][2][Imax][t] gate / up sums (slot 0: the shared expert)
  float* acc;               // ws: [t][h] block accumulator
  uint32_t* ftcount;        // ws: [slots][Imax / 128] K chunks added per feature tile
  uint32_t* hcount;         // ws: [h / 128] down blocks added per output tile
  DeviceStatus* st;
  int imax;                 // max(I, Is)
  int max_slots;            // 1 + min(E, t * k)
};

struct DfSmem {
  uint64_t full[D_NSLOT], empty[D_NSLOT];
  uint64_t a_full[D_NA], a_empty[D_NA];
  uint64_t acc_full[D_NACC], acc_empty[D_NACC];
  uint64_t hg_full[D_NHG], hg_empty[D_NHG];
  uint64_t ready;  // the routing is known (parts B, C, D)
  uint64_t esync;  // barrier of the four epilogue warps
  uint64_t drain;
  int32_t idx[D_MAX_PAIRS];
  float w[D_MAX_PAIRS];
  int32_t cnt[D_MAX_E + 1];
  int32_t off[D_MAX_E + 1];
  int32_t rows[D_MAX_PAIRS];
  float wts[D_MAX_PAIRS];
  int32_t slot_e[D_MAX_PAIRS + 1];     // expert of slot s >= 1 (slot 0: the shared expert)
  int32_t slot_row0[D_MAX_PAIRS + 1];  // first list position of slot s >= 1
  int32_t slot_n[D_MAX_PAIRS + 1];     // rows of slot s
  int32_t htcnt[D_MAX_H / 128];
  int32_t htlast[D_MAX_H / 128];
  int32_t wsum[4];
  int32_t n_touched;
  uint32_t tmem_slot;
  int abort;
};

constexpr size_t D_XT_BYTES = (size_t)(D_MAX_H / D_KC) * D_TILE;
constexpr size_t df_smem_bytes() {
  return 1024 + (size_t)D_NSLOT * D_SLOT + D_XT_BYTES + (size_t)D_NHG * D_TILE + sizeof(DfSmem);
}

__device__ __forceinline__ void df_timeout(DeviceStatus* st, volatile int* abort, uint32_t site) {
  if (atomicOr(&st->flags, FLAG_TIMEOUT) == 0) st->timeout_site = site;
  *abort = 1;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Spin (bounded) until *p >= target; false when it gave up or *abort is set.
__device__ __forceinline__ bool spin_until(const uint32_t* p, uint32_t target, const volatile int* abort) {
  if (ld_acquire(p) >= target) return true;
  const uint64_t t0 = globaltimer();
  for (;;) {
    __nanosleep(32);
    if (ld_acquire(p) >= target) return true;
    if (*abort || globaltimer() - t0 > D_WAIT_NS) return false;
  }
}

__device__ __forceinline__ void df_bulk(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// One item of this CTA's list: a gate/up block pair (a = feature tile, b =
// K chunk) or a down block (a = K chunk of inter, b = 128-row tile of h).
struct Item {
  int slot, a, b;
  bool gu;
};

// The CTA's list: A [0, nA) shared gate/up, B routed gate/up, C shared down,
// D routed down.  Routed slots are 1.. in expert order and all the same size.
struct Plan {
  int nkc, nht;
  int sa0, nA, rb0, nB, sc0, nC, rd0, nD;
  int per_gu, per_dn;  // blocks of one routed slot
  __device__ __forceinline__ int total() const { return nA + nB + nC + nD; }
  __device__ __forceinline__ Item at(int i) const {
    Item it;
    if (i < nA) {
      const int g = sa0 + i;
      it.slot = 0, it.a = g / nkc, it.b = g % nkc, it.gu = true;
    } else if (i < nA + nB) {
      const int g = rb0 + (i - nA);
      const int rel = g % per_gu;
      it.slot = 1 + g / per_gu, it.a = rel / nkc, it.b = rel % nkc, it.gu = true;
    } else if (i < nA + nB + nC) {
      const int g = sc0 + (i - nA - nB);
      it.slot = 0, it.a = g / nht, it.b = g % nht, it.gu = false;
    } else {
      const int g = rd0 + (i - nA - nB - nC);
      const int rel = g % per_dn;
      it.slot = 1 + g / per_dn, it.a = rel / nht, it.b = rel % nht, it.gu = false;
    }
    return it;
  }
  // Whether item i closes its gate/up segment (the next item is not a
  // gate/up pair of the same slot and feature tile) or its down chunk.
  __device__ __forceinline__ bool closes(int i) const {
    if (i + 1 >= total()) return true;
    const Item a = at(i), b = at(i + 1);
    return a.gu != b.gu || a.slot != b.slot || a.a != b.a;
  }
  __device__ __forceinline__ bool opens(int i) const {
    if (i == 0) return true;
    const Item a = at(i - 1), b = at(i);
    return a.gu != b.gu || a.slot != b.slot || a.a != b.a;
  }
};

__device__ __forceinline__ int split(int n, int b, int G) { return (int)((long)n * b / G); }

template <int NQ>
__global__ void __launch_bounds__(D_THREADS, 1) decode_fused_kernel(DfParams P) {
  extern __shared__ uint8_t df_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(df_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* xt = ring + (size_t)D_NSLOT * D_SLOT;  // x: h / 64 swizzled 16-row tiles
  uint8_t* hgt = xt + D_XT_BYTES;                 // silu(gate) * up tiles
  DfSmem& S = *reinterpret_cast<DfSmem*>(hgt + (size_t)D_NHG * D_TILE);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x, b = blockIdx.x;
  const int t = P.t, h = P.h, E = P.E, k = P.k;
  volatile int* abort = &S.abort;

  Plan L{};
  L.nkc = h / D_KC, L.nht = h / 128;
  L.per_gu = (P.I / 128) * L.nkc, L.per_dn = (P.I / D_KC) * L.nht;
  {
    const int sg = P.Is > 0 ? (P.Is / 128) * L.nkc : 0, sd = P.Is > 0 ? (P.Is / D_KC) * L.nht : 0;
    L.sa0 = split(sg, b, G), L.nA = split(sg, b + 1, G) - L.sa0;
    L.sc0 = split(sd, b, G), L.nC = split(sd, b + 1, G) - L.sc0;
    L.nB = 0, L.nD = 0, L.rb0 = 0, L.rd0 = 0;  // known after the routing
  }

  if (tid == 0) {
    for (int i = 0; i < D_NSLOT; ++i) mbar_init(&S.full[i], 1), mbar_init(&S.empty[i], 4);
    for (int i = 0; i < D_NA; ++i) mbar_init(&S.a_full[i], 4), mbar_init(&S.a_empty[i], 1);
    for (int i = 0; i < D_NACC; ++i) mbar_init(&S.acc_full[i], 1), mbar_init(&S.acc_empty[i], 4);
    for (int i = 0; i < D_NHG; ++i) mbar_init(&S.hg_full[i], 4), mbar_init(&S.hg_empty[i], 1);
    mbar_init(&S.ready, 1);
    mbar_init(&S.esync, 4);
    mbar_init(&S.drain, 1);
    S.abort = 0;
    fence_mbar_init();
  }
  // x into the swizzled B tiles (rows past t are zero)
  for (int q = tid; q < 16 * (h / 8); q += blockDim.x) {
    const int r = q / (h / 8), p = q % (h / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < t) v = __ldg(reinterpret_cast<const uint4*>(P.x + (size_t)r * h) + p);
    *reinterpret_cast<uint4*>(xt + (size_t)(p >> 3) * D_TILE + sw128_off(r, p & 7)) = v;
  }
  fence_async_smem();
  if (warp == W_ISSUE) tmem_alloc(&S.tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_slot;

  // The roles that start on part A wait here for parts B, C, D.
  auto await_plan = [&]() -> bool {
    if (!mbar_wait(&S.ready, 0, abort, D_WAIT_NS)) return false;
    if (*abort) return false;
    const int n = S.n_touched;
    const int rg = n * L.per_gu, rd = n * L.per_dn;
    L.rb0 = split(rg, b, G), L.nB = split(rg, b + 1, G) - L.rb0;
    L.rd0 = split(rd, b, G), L.nD = split(rd, b + 1, G) - L.rd0;
    return true;
  };

  if (warp == W_PROD) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      bool planned = false;
      int issued = 0;
      for (int i = 0; !*abort; ++i) {
        if (i == L.nA && !planned) {
          if (!await_plan()) break;
          planned = true;
        }
        if (i >= L.total()) break;
        const Item it = L.at(i);
        const int sl = i % D_NSLOT;
        if (!mbar_wait(&S.empty[sl], ((i / D_NSLOT) & 1) ^ 1, abort, D_WAIT_NS)) {
          df_timeout(P.st, abort, 71);
          break;
        }
        const int Iu = it.slot == 0 ? P.Is : P.I;
        const uint8_t* rec =
            it.slot == 0 ? P.s_packed : P.packed + (size_t)S.slot_e[it.slot] * packed_rec_bytes(h, P.I);
        const uint8_t* src;
        uint32_t bytes;
        if (it.gu) {
          src = rec + ((size_t)it.a * L.nkc + it.b) * D_SLOT;  // [feature tile][chunk][gate][up]
          bytes = D_SLOT;
        } else {
          src = rec + packed_gu_bytes(h, Iu) + ((size_t)it.b * (Iu / D_KC) + it.a) * PACK_QB;  // [out tile][chunk]
          bytes = PACK_QB;
        }
        mbar_arrive_expect_tx(&S.full[sl], bytes);
        df_bulk(ring + (size_t)sl * D_SLOT, src, bytes, &S.full[sl]);
        issued = i + 1;
      }
      if (*abort) {
        const int never = 0;  // let the last copy into every slot land
        for (int i = issued > D_NSLOT ? issued - D_NSLOT : 0; i < issued; ++i)
          mbar_wait(&S.full[i % D_NSLOT], (i / D_NSLOT) & 1, &never, 100000000ull);
      }
    }
  } else if (warp == W_ISSUE) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, 16);
      bool planned = false;
      uint32_t u = 0, hgi = 0;  // accumulation units (segments, down items), down chunks
      for (int i = 0; !*abort; ++i) {
        if (i == L.nA && !planned) {
          if (!await_plan()) break;
          planned = true;
        }
        if (i >= L.total()) break;
        const Item it = L.at(i);
        const int as = i % D_NA, ab = (int)(u % D_NACC);
        // the segment after part A always opens anew (another slot, or a down
        // block), so the close of part A is known before the routing
        const bool closes = (i + 1 == L.nA && !planned) ? true : L.closes(i);
        const bool opens = L.opens(i);
        if (opens || !it.gu) {
          if (!mbar_wait(&S.acc_empty[ab], ((u / D_NACC) & 1) ^ 1, abort, D_WAIT_NS)) {
            df_timeout(P.st, abort, 72);
            break;
          }
        }
        const int hs = (int)(hgi % D_NHG);
        if (!it.gu && opens) {
          if (!mbar_wait(&S.hg_full[hs], (hgi / D_NHG) & 1, abort, D_WAIT_NS)) {
            df_timeout(P.st, abort, 73);
            break;
          }
        }
        if (!mbar_wait(&S.a_full[as], (i / D_NA) & 1, abort, D_WAIT_NS)) {
          df_timeout(P.st, abort, 74);
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem + D_ACC_COL + ab * 32, a_st = tmem + as * 64;
        if (it.gu) {
          const uint64_t bd = desc_sw128(smem_u32(xt + (size_t)it.b * D_TILE));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t accum = (opens && kk == 0) ? 0u : 1u;
            mma_bf16_ta(acc, a_st + 8 * kk, bd + 2 * kk, idesc, accum);
            mma_bf16_ta(acc + 16, a_st + 32 + 8 * kk, bd + 2 * kk, idesc, accum);
          }
        } else {
          const uint64_t bd = desc_sw128(smem_u32(hgt + (size_t)hs * D_TILE));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) mma_bf16_ta(acc, a_st + 8 * kk, bd + 2 * kk, idesc, kk != 0);
        }
        mma_commit(&S.a_empty[as]);
        if (closes || !it.gu) {
          mma_commit(&S.acc_full[ab]);
          ++u;
        }
        if (!it.gu && closes) {
          mma_commit(&S.hg_empty[hs]);
          ++hgi;
        }
      }
      if (*abort) {
        mma_commit(&S.drain);
        const int never = 0;
        mbar_wait(&S.drain, 0, &never, 100000000ull);
      }
    }
  } else if (warp < W_EPI0) {
    // ---------------------------------------------------------------- dequantisation (two groups, alternate items)
    const int grp = (warp - W_DQ0) >> 2;
    const int q = warp & 3;       // tensor-memory lane quarter of this warp
    const int o = q * 32 + lane;  // weight row = tensor-memory lane
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    bool planned = false;
    for (int i = grp; !*abort; i += 2) {
      if (i >= L.nA && !planned) {
        if (!__all_sync(0xFFFFFFFFu, await_plan())) break;
        planned = true;
      }
      if (i >= L.total()) break;
      const Item it = L.at(i);
      const int sl = i % D_NSLOT, as = i % D_NA;
      const bool got = mbar_wait(&S.full[sl], (i / D_NSLOT) & 1, abort, D_WAIT_NS) &&
                       mbar_wait(&S.a_empty[as], ((i / D_NA) & 1) ^ 1, abort, D_WAIT_NS);
      if (!__all_sync(0xFFFFFFFFu, got)) {
        if (lane == 0) df_timeout(P.st, abort, 75);
        break;
      }
      tc_fence_after();
      const uint8_t* blk = ring + (size_t)sl * D_SLOT;
      const int nblk = it.gu ? 2 : 1;
      for (int m = 0; m < nblk; ++m) {
        const uint8_t* bm = blk + m * PACK_QB;
        const __nv_bfloat16 sv = reinterpret_cast<const __nv_bfloat16*>(bm + 4096)[o];
        const __nv_bfloat16 bv = reinterpret_cast<const __nv_bfloat16*>(bm + 4096 + 256)[o];
        const uint4 c0 = reinterpret_cast<const uint4*>(bm + o * 32)[0];
        const uint4 c1 = reinterpret_cast<const uint4*>(bm + o * 32)[1];
        const uint32_t wd[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        uint32_t r[32];
        dequant_packed<8>(wd, __halves2bfloat162(sv, sv), __halves2bfloat162(bv, bv), r);
        tmem_st<32>(lane_base + as * 64 + m * 32, r);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&S.a_full[as]);
        mbar_arrive(&S.empty[sl]);  // the codes are in tensor memory: the ring slot is free
      }
    }
  } else {
    // ---------------------------------------------------------------- router, grouping, epilogue
    const int ew = warp - W_EPI0;  // 0..3
    const int etid = tid - W_EPI0 * 32;
    uint32_t ephase = 0;
    // barrier of the four epilogue warps, bounded
    auto esync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.esync);
      const bool got = __all_sync(0xFFFFFFFFu, mbar_wait(&S.esync, ephase, abort, D_WAIT_NS));
      ephase ^= 1u;
      if (!got && lane == 0) df_timeout(P.st, abort, 76);
      return got;
    };

    // 1. router logits (experts b, b + G, ...), the shared gate, zeroing
    {
      const int nm = (h + 255) / 256;
      for (int e = b; e < E; e += G) {
        const uint16_t* wrow = P.wr + (size_t)e * h;
        for (int r = ew; r < t; r += 4) {
          const uint16_t* xr = P.x + (size_t)r * h;
          float a = 0.f;
          for (int m0 = 0; m0 < nm; m0 += 8) {
            uint4 wv[8], xv[8];  // every load of the batch in flight together
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int k0 = (m0 + u) * 256 + lane * 8;
              const bool in = m0 + u < nm && k0 < h;
              wv[u] = in ? __ldg(reinterpret_cast<const uint4*>(wrow + k0)) : make_uint4(0, 0, 0, 0);
              xv[u] = in ? __ldg(reinterpret_cast<const uint4*>(xr + k0)) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              if (m0 + u >= nm || (m0 + u) * 256 + lane * 8 >= h) continue;
#pragma unroll
              for (int cc = 0; cc < 8; ++cc) {
                const uint32_t ww = (&wv[u].x)[cc >> 1], xw = (&xv[u].x)[cc >> 1];
                a = fmaf((cc & 1) ? bf16hi(xw) : bf16lo(xw), (cc & 1) ? bf16hi(ww) : bf16lo(ww), a);
              }
            }
          }
          a = a + __shfl_xor_sync(0xFFFFFFFFu, a, 16);
          a = a + __shfl_xor_sync(0xFFFFFFFFu, a, 8);
          a = a + __shfl_xor_sync(0xFFFFFFFFu, a, 4);
          a = a + __shfl_xor_sync(0xFFFFFFFFu, a, 2);
          a = a + __shfl_xor_sync(0xFFFFFFFFu, a, 1);
          if (lane == 0) P.logits[(size_t)r * P.Ep + e] = P.rbias ? a + P.rbias[e] : a;
        }
      }
      if (P.s_gate && b == G - 1) {
        for (int r = ew; r < t; r += 4) {
          float s = 0.f;
          for (int i = lane; i < h; i += 32) s = fmaf(bf16f(P.x[(size_t)r * h + i]), bf16f(P.s_gate[i]), s);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
          if (lane == 0) P.gate_vals[r] = 1.f / (1.f + __expf(-s));
        }
      }
      const size_t n_gu = (size_t)P.max_slots * 2 * P.imax * t, n_acc = (size_t)t * h;
      const size_t n_ft = (size_t)P.max_slots * (P.imax / 128), n_h = (size_t)h / 128;
      const size_t gt = (size_t)b * 128 + etid, gs = (size_t)G * 128;
      for (size_t i = gt; i < n_gu; i += gs) P.gu[i] = 0.f;
      for (size_t i = gt; i < n_acc; i += gs) P.acc[i] = 0.f;
      for (size_t i = gt; i < n_ft; i += gs) P.ftcount[i] = 0u;
      for (size_t i = gt; i < n_h; i += gs) P.hcount[i] = 0u;
    }
    // grid-wide barrier: every call advances the counter by G, so the target
    // is the next multiple of G above this CTA's arrival
    __threadfence();
    bool ok = esync();
    if (ok && etid == 0) {
      const uint32_t arrival = atomicAdd(&P.st->fused_bar, 1u);
      const uint32_t target = (arrival / (uint32_t)G + 1u) * (uint32_t)G;
      if (!spin_until(&P.st->fused_bar, target, abort)) df_timeout(P.st, abort, 77);
    }
    ok = esync() && !*abort;

    // 2. selection and grouping (every CTA; E <= 256, t * k <= 128)
    if (ok) {
      for (int r = ew; r < t; r += 4) {
        uint64_t key[NQ];
#pragma unroll
        for (int qq = 0; qq < NQ; ++qq) {
          const int e = lane + 32 * qq;
          key[qq] = e < E ? topk_key(__ldcg(P.logits + (size_t)r * P.Ep + e), e) : 0ull;
        }
        warp_topk_softmax<NQ>(key, k, lane, S.idx + r * k, S.w + r * k);
      }
      for (int e = etid; e <= E; e += 128) S.cnt[e] = 0;
      ok = esync();
    }
    const int npairs = t * k;
    if (ok) {
      for (int p = etid; p < npairs; p += 128) atomicAdd(&S.cnt[S.idx[p]], 1);
      ok = esync();
    }
    if (ok) {
      // scan over the experts, two per thread: list offsets and the slot of
      // every touched expert
      const int e0 = 2 * etid, e1 = e0 + 1;
      const int n0 = e0 < E ? S.cnt[e0] : 0, n1 = e1 < E ? S.cnt[e1] : 0;
      const int u0 = n0 > 0, u1 = n1 > 0;
      int sn = n0 + n1, su = u0 + u1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int yn = __shfl_up_sync(0xFFFFFFFFu, sn, o), yu = __shfl_up_sync(0xFFFFFFFFu, su, o);
        if (lane >= o) sn += yn, su += yu;
      }
      if (lane == 31) S.wsum[ew] = (sn << 16) | su;
      ok = esync();
      if (ok) {
        int bn = 0, bu = 0;
        for (int qq = 0; qq < ew; ++qq) bn += S.wsum[qq] >> 16, bu += S.wsum[qq] & 0xFFFF;
        const int off0 = bn + sn - n0 - n1, s0 = bu + su - u0 - u1;
        if (e0 < E) {
          S.off[e0] = off0;
          if (u0) S.slot_e[1 + s0] = e0, S.slot_row0[1 + s0] = off0, S.slot_n[1 + s0] = n0;
        }
        if (e1 < E) {
          S.off[e1] = off0 + n0;
          if (u1) S.slot_e[1 + s0 + u0] = e1, S.slot_row0[1 + s0 + u0] = off0 + n0, S.slot_n[1 + s0 + u0] = n1;
        }
        if (etid == 127) {
          S.off[E] = bn + sn;
          S.n_touched = bu + su;
          S.slot_n[0] = t;
        }
        ok = esync();
      }
    }
    if (ok) {
      // stable placement: within an expert, rows ascend (a row names an expert once)
      for (int p = etid; p < npairs; p += 128) {
        const int e = S.idx[p], r = p / k;
        int rank = 0;
        for (int qq = 0; qq < r * k; ++qq) rank += S.idx[qq] == e;
        const int pos = S.off[e] + rank;
        S.rows[pos] = r;
        S.wts[pos] = S.w[p];
        if (b == 0) P.csr.slot_of[p] = pos;
      }
      for (int i = etid; i < h / 128; i += 128) S.htcnt[i] = 0;
      ok = esync();
    }
    if (ok && b == 0) {
      for (int p = etid; p < npairs; p += 128) {
        P.idx[p] = S.idx[p];
        P.w[p] = S.w[p];
        P.csr.rows[p] = S.rows[p];
        P.csr.weights[p] = S.wts[p];
      }
      for (int e = etid; e <= E; e += 128) P.csr.offsets[e] = S.off[e];
    }
    // parts B, C, D are known: release the other roles (an abort releases
    // them too; they read the flag)
    if (etid == 0) mbar_arrive(&S.ready);
    ok = ok && __all_sync(0xFFFFFFFFu, await_plan());

    // 3. epilogue: drain the accumulators in item order
    const int qd = warp & 3;  // tensor-memory lane quarter of this warp
    const uint32_t lane_base = tmem + ((uint32_t)(qd * 32) << 16);
    uint32_t u = 0, hgi = 0;
    int seg_n = 0;
    for (int i = 0; ok && i < L.total(); ++i) {
      const Item it = L.at(i);
      const bool closes = L.closes(i), opens = L.opens(i);
      const int n_tok = S.slot_n[it.slot];
      const int row0 = it.slot == 0 ? -1 : S.slot_row0[it.slot];
      if (it.gu) {
        ++seg_n;
        if (!closes) continue;
        const int ab = (int)(u % D_NACC);
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&S.acc_full[ab], (u / D_NACC) & 1, abort, D_WAIT_NS))) {
          if (lane == 0) df_timeout(P.st, abort, 78);
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t gv[16], uv[16];
        tmem_ld16(lane_base + D_ACC_COL + ab * 32, gv);
        tmem_ld16(lane_base + D_ACC_COL + ab * 32 + 16, uv);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.acc_empty[ab]);
        // column j of the accumulator is x row j; keep the slot's rows
        const int f = it.a * 128 + qd * 32 + lane;
        float* gb = P.gu + (size_t)it.slot * 2 * P.imax * t;
        for (int n = 0; n < n_tok; ++n) {
          const int r = row0 < 0 ? n : S.rows[row0 + n];
          float gval = 0.f, uval = 0.f;
#pragma unroll
          for (int j = 0; j < D_MAX_T; ++j)
            if (j == r) gval = __uint_as_float(gv[j]), uval = __uint_as_float(uv[j]);
          atomicAdd(gb + (size_t)f * t + n, gval);
          atomicAdd(gb + (size_t)(P.imax + f) * t + n, uval);
        }
        __threadfence();
        if (!esync()) {
          ok = false;
          break;
        }
        if (etid == 0) atomicAdd(&P.ftcount[(size_t)it.slot * (P.imax / 128) + it.a], (uint32_t)seg_n);
        seg_n = 0;
        ++u;
      } else {
        const int hs = (int)(hgi % D_NHG);
        if (opens) {
          // silu(gate) * up of this chunk for the slot's rows, once its
          // feature tile is complete
          bool got = true;
          if (lane == 0) got = mbar_wait(&S.hg_empty[hs], ((hgi / D_NHG) & 1) ^ 1, abort, D_WAIT_NS);
          if (etid == 0 && got) {
            got = spin_until(P.ftcount + (size_t)it.slot * (P.imax / 128) + it.a / 2, (uint32_t)L.nkc, abort);
            if (!got) df_timeout(P.st, abort, 79);
          }
          got = __shfl_sync(0xFFFFFFFFu, got, 0);
          if (!esync() || !got || *abort) {
            ok = false;
            break;
          }
          const float* gb = P.gu + (size_t)it.slot * 2 * P.imax * t;
          const int n = etid >> 3, pc = etid & 7;  // token row n of the tile, 16-byte piece pc
          uint32_t pk[4] = {0u, 0u, 0u, 0u};
          if (n < n_tok) {
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const int f = it.a * D_KC + pc * 8 + 2 * e2;
              const float v0 =
                  silu_mul_fast(__ldcg(gb + (size_t)f * t + n), __ldcg(gb + (size_t)(P.imax + f) * t + n));
              const float v1 = silu_mul_fast(__ldcg(gb + (size_t)(f + 1) * t + n),
                                             __ldcg(gb + (size_t)(P.imax + f + 1) * t + n));
              pk[e2] = ((uint32_t)f2bf(v1) << 16) | f2bf(v0);
            }
          }
          *reinterpret_cast<uint4*>(hgt + (size_t)hs * D_TILE + sw128_off(n, pc)) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
          fence_async_smem();  // the tensor core reads the tile through the async proxy
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.hg_full[hs]);
        }
        if (closes) ++hgi;
        const int ab = (int)(u % D_NACC);
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&S.acc_full[ab], (u / D_NACC) & 1, abort, D_WAIT_NS))) {
          if (lane == 0) df_timeout(P.st, abort, 80);
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t yv[16];
        tmem_ld16(lane_base + D_ACC_COL + ab * 32, yv);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.acc_empty[ab]);
        // column n is the slot's n-th row: weight * y into the block accumulator
        const int col = it.b * 128 + qd * 32 + lane;
#pragma unroll
        for (int n = 0; n < D_MAX_T; ++n) {
          if (n < n_tok) {
            int r;
            float wt;
            if (row0 < 0) {
              r = n;
              wt = P.s_gate ? P.gate_vals[n] : 1.f;
            } else {
              r = S.rows[row0 + n];
              wt = S.wts[row0 + n];
            }
            atomicAdd(P.acc + (size_t)r * h + col, wt * __uint_as_float(yv[n]));
          }
        }
        if (etid == 0) S.htcnt[it.b] += 1;
        ++u;
      }
    }

    // 4. output tiles this CTA completes (after every epilogue thread's additions)
    __threadfence();
    ok = esync() && ok && !*abort;
    if (ok) {
      const uint32_t per_tile = (uint32_t)(S.n_touched * (P.I / D_KC) + (P.Is > 0 ? P.Is / D_KC : 0));
      for (int ht = etid; ht < L.nht; ht += 128) {
        const int mine = S.htcnt[ht];
        S.htlast[ht] = mine > 0 && atomicAdd(&P.hcount[ht], (uint32_t)mine) + (uint32_t)mine == per_tile;
      }
      __threadfence();
      ok = esync();
    }
    if (ok) {
      for (int ht = 0; ht < L.nht; ++ht) {
        if (!S.htlast[ht]) continue;
        for (int qq = etid; qq < t * 128; qq += 128) {
          const int r = qq / 128, c = ht * 128 + qq % 128;
          P.out[(size_t)r * h + c] = f2bf(__ldcg(P.acc + (size_t)r * h + c));
        }
      }
    }
  }

  // every role has finished and its copies and MMAs have landed: free tensor memory
  tc_fence_before();
  __syncthreads();
  if (warp == W_ISSUE) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int NQ>
cudaError_t launch_df(const DfParams& P, cudaStream_t stream) {
  cudaError_t err = set_smem_limit_once(decode_fused_kernel<NQ>, (int)df_smem_bytes());
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sm_count());
  cfg.blockDim = dim3(D_THREADS);
  cfg.dynamicSmemBytes = df_smem_bytes();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: the grid barrier and counters need it
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  MOE_LAUNCH("decode_fused", stream, (err = cudaLaunchKernelEx(&cfg, decode_fused_kernel<NQ>, P)));
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace

bool decode_fused_ok(const moe_dims& d, uint32_t flags) {
  return d.t <= D_MAX_T && d.E <= D_MAX_E && d.h <= D_MAX_H && (flags & MOE_PACKED_WEIGHTS) &&
         (flags & MOE_FUSED_DECODE) &&
         !(flags & (MOE_DETERMINISTIC | MOE_FORCE_SMALL_T | MOE_FORCE_LARGE_T | MOE_SIMPLE_KERNELS));
}

size_t decode_fused_ws_bytes(const moe_dims& d) {
  const int imax = d.inter > d.shared_inter ? d.inter : d.shared_inter;
  const int slots = 1 + (d.E < d.t * d.k ? d.E : d.t * d.k);
  const int Ep = (d.E + 15) / 16 * 16;
  return align_up((size_t)d.t * Ep * 4, 256) + align_up((size_t)d.t * 4, 256) +
         align_up((size_t)slots * 2 * imax * d.t * 4, 256) + align_up((size_t)d.t * d.h * 4, 256) +
         align_up((size_t)slots * (imax / 128) * 4, 256) + align_up((size_t)(d.h / 128) * 4, 256);
}

cudaError_t launch_decode_fused(const uint16_t* x, const uint16_t* wr, const float* rbias, const moe_dims& d,
                                const uint8_t* packed, const uint8_t* s_packed, const uint16_t* s_gate, int32_t* idx,
                                float* w, const moe_csr& csr, uint16_t* out, unsigned char* scratch,
                                DeviceStatus* st, cudaStream_t stream) {
  DfParams P{};
  P.t = d.t, P.h = d.h, P.I = d.inter, P.Is = d.shared_inter, P.E = d.E, P.Ep = (d.E + 15) / 16 * 16, P.k = d.k;
  P.x = x, P.wr = wr, P.rbias = rbias, P.s_gate = d.shared_inter > 0 ? s_gate : nullptr;
  P.packed = packed, P.s_packed = s_packed;
  P.idx = idx, P.w = w, P.csr = csr, P.out = out;
  P.imax = d.inter > d.shared_inter ? d.inter : d.shared_inter;
  P.max_slots = 1 + (d.E < d.t * d.k ? d.E : d.t * d.k);
  unsigned char* q = scratch;
  auto take = [&](size_t bytes) {
    unsigned char* p = q;
    q += align_up(bytes, 256);
    return p;
  };
  P.logits = reinterpret_cast<float*>(take((size_t)d.t * P.Ep * 4));
  P.gate_vals = reinterpret_cast<float*>(take((size_t)d.t * 4));
  P.gu = reinterpret_cast<float*>(take((size_t)P.max_slots * 2 * P.imax * d.t * 4));
  P.acc = reinterpret_cast<float*>(take((size_t)d.t * d.h * 4));
  P.ftcount = reinterpret_cast<uint32_t*>(take((size_t)P.max_slots * (P.imax / 128) * 4));
  P.hcount = reinterpret_cast<uint32_t*>(take((size_t)(d.h / 128) * 4));
  P.st = st;
  const int NQ = (d.E + 31) / 32;
  if (NQ <= 1) return launch_df<1>(P, stream);
  if (NQ <= 2) return launch_df<2>(P, stream);
  if (NQ <= 4) return launch_df<4>(P, stream);
  return launch_df<8>(P, stream);
}

}  // namespace moe

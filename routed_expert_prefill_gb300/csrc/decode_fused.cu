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
// Gate/up pairs run [expert][feature tile][K chunk of h], down blocks
// [expert][output tile][K chunk of inter], so consecutive items of a CTA
// accumulate into one tensor-memory accumulator (a "segment") that is read
// out once, when the segment closes.  The CTA's list is written once into
// shared memory as packed (expert slot, tile, K chunk, open/close) entries:
// part A in the prologue, parts B to D as soon as the routing is known.
//
// Warp roles (14 warps):
//   0      producer: one thread bulk-copies the blocks of the CTA's items
//          into a ring in shared memory, starting with part A at once;
//   1      MMA issuer: the warp walks the list in step, one elected lane
//          issues tcgen05.mma (M = 128 weight rows, N = 16 token columns, A in
//          tensor memory, B in shared memory);
//   2-9    first x into shared memory, then two dequantisation groups taking
//          alternate items: one weight row per thread, w = fma(q, s, b) in
//          bf16 (one rounding) straight into tensor memory (tcgen05.st);
//   10-13  first the router: the logits of experts b, b + G, ... in the
//          fixed summation order of moe_route_topk (lane l owns
//          K = 256 m + 8 l + c, m then c ascending from +0, lane sums
//          combined by the xor butterfly 16..1, bias last), zeroing of the
//          accumulators, a grid-wide barrier (a generation counter every call
//          advances by the grid size), top-k and grouping (identical in every
//          CTA; CTA 0 writes idx, w and the CSR arrays), the rest of the list;
//          then the epilogue: tcgen05.ld of each closed segment and fp32
//          atomics into the per-expert gate/up sums or the block accumulator.
//
// Operands.  Gate/up: B is x, staged once as 64-wide K chunks of 16 rows
// (128-byte swizzled, rows past t zero), so every expert is multiplied with
// all t rows -- at N = 16 the MMA costs the same -- and the epilogue keeps
// the columns of the expert's own rows.  Down: B is silu(gate) * up of one
// 64-wide chunk for the expert's rows (rounded to bf16, as the hidden
// activations are everywhere else).  A counter per (expert, 128-row feature
// tile) counts the K chunks added; the CTA whose addition completes the tile
// writes its two B tiles to the workspace, already in the swizzled layout,
// and raises the tile's flag; the producer waits for the flag before it
// bulk-copies a down block together with its B tile into one ring slot.  A
// counter per 128-column output tile lets the last contributor round the
// tile to bf16.
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
constexpr int D_SLOT = 2 * PACK_QB;  // ring slot: a gate/up block pair, or a down block and its B tile
constexpr int D_HG_OFF = 5 * 1024;   // the B tile of a down item within its slot (1024-byte aligned)
constexpr int D_NSLOT = 12;
constexpr int D_NA = 4;              // tensor-memory A slots of 64 columns (a gate/up pair, or a down block)
constexpr int D_NACC = 8;            // accumulator buffers of 32 columns (gate 16 + up 16, or down 16)
constexpr int D_ACC_COL = D_NA * 64;
constexpr int D_TILE = 2048;         // 16 rows x 128 bytes, swizzled
constexpr int D_MAX_H = 2048;        // x is staged as h / 64 tiles
constexpr int D_MAX_T = 8;
constexpr int D_MAX_E = 256;
constexpr int D_MAX_PAIRS = D_MAX_T * 16;
constexpr int D_MAX_ITEMS = 2048;    // entries of a CTA's list
constexpr int D_KC = 64;
constexpr uint64_t D_WAIT_NS = 2000000000ull;
static_assert(PACK_QB <= D_HG_OFF && D_HG_OFF + D_TILE <= D_SLOT, "down item layout in a ring slot");
static_assert(D_SLOT % 1024 == 0, "ring slots keep the 1024-byte alignment of the swizzled tiles");

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
  float* gu;                // ws: [t + t * k][2][Imax] gate / up sums: rows of the shared expert, then list positions
  float* acc;               // ws: [t][h] block accumulator
  uint32_t* ftcount;        // ws: [slots][Imax / 128] K chunks added per feature tile
  uint32_t* hgready;        // ws: [slots] feature tiles whose B tiles are written
  uint8_t* hg;              // ws: [slots][Imax / 64] swizzled bf16 B tiles of the down pass
  uint32_t* hcount;         // ws: [h / 128] down blocks added per output tile
  DeviceStatus* st;
  int imax;                 // max(I, Is)
  int max_slots;            // 1 + min(E, t * k)
};

struct DfSmem {
  uint64_t full[D_NSLOT], empty[D_NSLOT];
  uint64_t a_full[D_NA], a_empty[D_NA];
  uint64_t acc_full[D_NACC], acc_empty[D_NACC];
  uint64_t x_ready;  // x is in its B tiles
  uint64_t ready;    // the routing is known: parts B, C, D are in the list
  uint64_t esync;    // barrier of the four epilogue warps
  uint64_t drain;
  uint32_t items[D_MAX_ITEMS];
  int32_t idx[D_MAX_PAIRS];
  float w[D_MAX_PAIRS];
  int32_t cnt[D_MAX_E];
  int32_t off[D_MAX_E + 1];
  int32_t rows[D_MAX_PAIRS];
  float wts[D_MAX_PAIRS];
  int32_t slot_e[D_MAX_PAIRS + 1];     // expert of slot s >= 1 (slot 0: the shared expert)
  int32_t slot_row0[D_MAX_PAIRS + 1];  // first list position of slot s >= 1
  int32_t slot_n[D_MAX_PAIRS + 1];     // rows of slot s
  int32_t htcnt[D_MAX_H / 128];
  int32_t htlast[D_MAX_H / 128];
  int32_t n_items;  // entries in the list (part A alone until `ready`)
  int32_t n_touched;
  int32_t last;     // this CTA completed the feature tile just drained
  uint32_t tmem_slot;
  int abort;
};

constexpr size_t D_XT_BYTES = (size_t)(D_MAX_H / D_KC) * D_TILE;
constexpr size_t df_smem_bytes() { return 1024 + (size_t)D_NSLOT * D_SLOT + D_XT_BYTES + sizeof(DfSmem); }

__device__ __forceinline__ void df_timeout(DeviceStatus* st, volatile int* abort, uint32_t site) {
  if (atomicOr(&st->flags, FLAG_TIMEOUT) == 0) st->timeout_site = site;
  *abort = 1;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Orders this thread's generic-proxy global accesses with its bulk copies.
__device__ __forceinline__ void fence_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

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

// A list entry: expert slot (0: the shared expert), tile (gate/up: 128-row
// feature tile; down: 128-column output tile), K chunk (gate/up: of h; down:
// of inter), and whether the item opens / closes its segment.
struct Item {
  int slot, tile, kc;
  bool gu, opens, closes;
};
__device__ __forceinline__ Item item_unpack(uint32_t v) {
  Item it;
  it.slot = (int)(v & 0xFFu), it.tile = (int)((v >> 8) & 0xFFu), it.kc = (int)((v >> 16) & 0xFFu);
  it.gu = (v >> 24) & 1u, it.opens = (v >> 25) & 1u, it.closes = (v >> 26) & 1u;
  return it;
}

// The CTA's ranges of the four parts.  Routed slots are 1.. in expert order
// and all the same size.
struct Plan {
  int nkc, nht;        // K chunks of h, 128-column tiles of h
  int nkd_s, nkd_r;    // K chunks of the down pass: Is / 64, I / 64
  int per_gu, per_dn;  // items of one routed slot
  int sa0, nA, rb0, nB, sc0, nC, rd0, nD;
  __device__ __forceinline__ int total() const { return nA + nB + nC + nD; }
  // Entry of item i.  Within a part, item g covers (slot base + g / per,
  // tile (g % per) / n, K chunk g % n); a segment is a run of K chunks of one
  // (slot, tile), so it opens at K chunk 0 or at the part's first item and
  // closes at K chunk n - 1 or at the part's last item.  Neighbours from
  // different parts are always in different segments (the pass or the slot
  // differs), so the close of part A is known before the routing.
  __device__ __forceinline__ uint32_t entry(int i) const {
    int gu, s0, per, n, g0, cnt;
    if (i < nA) {
      gu = 1, s0 = 0, per = 0x7FFFFFFF, n = nkc, g0 = sa0, cnt = nA;
    } else if ((i -= nA) < nB) {
      gu = 1, s0 = 1, per = per_gu, n = nkc, g0 = rb0, cnt = nB;
    } else if ((i -= nB) < nC) {
      gu = 0, s0 = 0, per = 0x7FFFFFFF, n = nkd_s, g0 = sc0, cnt = nC;
    } else {
      i -= nC;
      gu = 0, s0 = 1, per = per_dn, n = nkd_r, g0 = rd0, cnt = nD;
    }
    const int g = g0 + i, sl = g / per, rel = g - sl * per, tile = rel / n, kc = rel - tile * n;
    const bool opens = kc == 0 || i == 0, closes = kc == n - 1 || i == cnt - 1;
    return (uint32_t)(s0 + sl) | ((uint32_t)tile << 8) | ((uint32_t)kc << 16) | ((uint32_t)gu << 24) |
           ((uint32_t)opens << 25) | ((uint32_t)closes << 26);
  }
};

__device__ __forceinline__ int split(int n, int b, int G) { return (int)((long)n * b / G); }

template <int NQ>
__global__ void __launch_bounds__(D_THREADS, 1) decode_fused_kernel(DfParams P) {
  extern __shared__ uint8_t df_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(df_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* xt = ring + (size_t)D_NSLOT * D_SLOT;  // x: h / 64 swizzled 16-row tiles
  DfSmem& S = *reinterpret_cast<DfSmem*>(xt + D_XT_BYTES);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x, b = blockIdx.x;
  const int t = P.t, h = P.h, E = P.E, k = P.k;
  volatile int* abort = &S.abort;

  Plan L{};
  L.nkc = h / D_KC, L.nht = h / 128;
  L.nkd_s = P.Is / D_KC, L.nkd_r = P.I / D_KC;
  L.per_gu = (P.I / 128) * L.nkc, L.per_dn = L.nht * L.nkd_r;
  {
    const int sg = (P.Is / 128) * L.nkc, sd = L.nht * L.nkd_s;
    L.sa0 = split(sg, b, G), L.nA = split(sg, b + 1, G) - L.sa0;
    L.sc0 = split(sd, b, G), L.nC = split(sd, b + 1, G) - L.sc0;
    L.nB = 0, L.nD = 0, L.rb0 = 0, L.rd0 = 0;  // known after the routing
  }
  if (tid == 0) {
    for (int i = 0; i < D_NSLOT; ++i) mbar_init(&S.full[i], 1), mbar_init(&S.empty[i], 1);
    for (int i = 0; i < D_NA; ++i) mbar_init(&S.a_full[i], 4), mbar_init(&S.a_empty[i], 1);
    for (int i = 0; i < D_NACC; ++i) mbar_init(&S.acc_full[i], 1), mbar_init(&S.acc_empty[i], 4);
    mbar_init(&S.x_ready, 8);
    mbar_init(&S.ready, 1);
    mbar_init(&S.esync, 4);
    mbar_init(&S.drain, 1);
    S.abort = 0;
    S.n_items = L.nA;
    fence_mbar_init();
  }
  for (int i = tid; i < L.nA; i += D_THREADS) S.items[i] = L.entry(i);
  if (warp == W_ISSUE) tmem_alloc(&S.tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_slot;

  // The roles that start on part A wait here for parts B, C, D; the list's
  // length comes back (0 after an abort).
  auto await_plan = [&]() -> int {
    if (!mbar_wait(&S.ready, 0, abort, D_WAIT_NS)) return 0;
    return *abort ? 0 : S.n_items;
  };

  if (warp == W_PROD) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int total = L.nA, issued = 0;
      bool planned = false;
      int hg_slot = -1;
      const size_t rec_bytes = packed_rec_bytes(h, P.I);
      const int kd_per_slot = P.imax / D_KC;
      for (int i = 0; !*abort; ++i) {
        if (i == total && !planned) {
          total = await_plan();
          planned = true;
        }
        if (i >= total) break;
        const Item it = item_unpack(S.items[i]);
        const int sl = i % D_NSLOT;
        if (!mbar_wait(&S.empty[sl], ((i / D_NSLOT) & 1) ^ 1, abort, D_WAIT_NS)) {
          df_timeout(P.st, abort, 71);
          break;
        }
        const uint8_t* rec = it.slot == 0 ? P.s_packed : P.packed + (size_t)S.slot_e[it.slot] * rec_bytes;
        uint8_t* dst = ring + (size_t)sl * D_SLOT;
        if (it.gu) {
          mbar_arrive_expect_tx(&S.full[sl], D_SLOT);
          df_bulk(dst, rec + ((size_t)it.tile * L.nkc + it.kc) * D_SLOT, D_SLOT, &S.full[sl]);  // [ftile][chunk][g][u]
        } else {
          const int Iu = it.slot == 0 ? P.Is : P.I;
          if (it.slot != hg_slot) {  // every B tile of the slot is written once all its feature tiles are complete
            if (!spin_until(P.hgready + it.slot, (uint32_t)(Iu / 128), abort)) {
              df_timeout(P.st, abort, 70);
              break;
            }
            fence_async_global();
            hg_slot = it.slot;
          }
          mbar_arrive_expect_tx(&S.full[sl], PACK_QB + D_TILE);
          df_bulk(dst, rec + packed_gu_bytes(h, Iu) + ((size_t)it.tile * (Iu / D_KC) + it.kc) * PACK_QB, PACK_QB,
                  &S.full[sl]);  // [out tile][chunk]
          df_bulk(dst + D_HG_OFF, P.hg + ((size_t)it.slot * kd_per_slot + it.kc) * D_TILE, D_TILE, &S.full[sl]);
        }
        issued = i + 1;
      }
      if (*abort) {
        const int never = 0;  // let the last copy into every slot land
        for (int i = issued > D_NSLOT ? issued - D_NSLOT : 0; i < issued; ++i)
          mbar_wait(&S.full[i % D_NSLOT], (i / D_NSLOT) & 1, &never, 100000000ull);
      }
    }
  } else if (warp == W_ISSUE) {
    // ---------------------------------------------------------------- MMA issuer (warp-uniform)
    const uint32_t idesc = idesc_bf16(128, 16);
    int total = L.nA;
    bool planned = false, live = true;
    uint32_t u = 0;  // segments
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(&S.x_ready, 0, abort, D_WAIT_NS))) {
      if (lane == 0) df_timeout(P.st, abort, 69);
      live = false;
    }
    for (int i = 0; live && !__any_sync(0xFFFFFFFFu, *abort); ++i) {  // warp-uniform exit
      if (i == total && !planned) {
        total = __shfl_sync(0xFFFFFFFFu, await_plan(), 0);
        planned = true;
      }
      if (i >= total) break;
      const Item it = item_unpack(S.items[i]);
      const int as = i % D_NA, sl = i % D_NSLOT, ab = (int)(u % D_NACC);
      bool got = true;
      if (it.opens) got = mbar_wait(&S.acc_empty[ab], ((u / D_NACC) & 1) ^ 1, abort, D_WAIT_NS);
      got = got && mbar_wait(&S.a_full[as], (i / D_NA) & 1, abort, D_WAIT_NS);
      if (!__all_sync(0xFFFFFFFFu, got)) {
        if (lane == 0) df_timeout(P.st, abort, 74);
        break;
      }
      if (elect_one()) {
        tc_fence_after();
        const uint32_t acc = tmem + D_ACC_COL + ab * 32, a_st = tmem + as * 64;
        if (it.gu) {
          const uint64_t bd = desc_sw128(smem_u32(xt + (size_t)it.kc * D_TILE));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t accum = (it.opens && kk == 0) ? 0u : 1u;
            mma_bf16_ta(acc, a_st + 8 * kk, bd + 2 * kk, idesc, accum);
            mma_bf16_ta(acc + 16, a_st + 32 + 8 * kk, bd + 2 * kk, idesc, accum);
          }
        } else {
          const uint64_t bd = desc_sw128(smem_u32(ring + (size_t)sl * D_SLOT + D_HG_OFF));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ta(acc, a_st + 8 * kk, bd + 2 * kk, idesc, (it.opens && kk == 0) ? 0u : 1u);
        }
        mma_commit(&S.a_empty[as]);
        mma_commit(&S.empty[sl]);  // the codes (and a down item's B tile) are consumed
        if (it.closes) mma_commit(&S.acc_full[ab]);
      }
      __syncwarp();
      if (it.closes) ++u;
    }
    if (__any_sync(0xFFFFFFFFu, *abort) && elect_one()) {
      mma_commit(&S.drain);
      const int never = 0;
      mbar_wait(&S.drain, 0, &never, 100000000ull);
    }
    __syncwarp();
  } else if (warp < W_EPI0) {
    // ---------------------------------------------------------------- x, then dequantisation
    {
      // x into the swizzled B tiles (rows past t are zero), the loads of a
      // batch in flight together
      const int dtid = tid - W_DQ0 * 32, hp = h / 8, nq = 16 * hp;
      for (int q0 = dtid; q0 < nq; q0 += 256 * 8) {
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int q = q0 + j * 256, r = q / hp, p = q - r * hp;
          v[j] = (q < nq && r < t) ? __ldg(reinterpret_cast<const uint4*>(P.x + (size_t)r * h) + p)
                                   : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int q = q0 + j * 256, r = q / hp, p = q - r * hp;
          if (q < nq) *reinterpret_cast<uint4*>(xt + (size_t)(p >> 3) * D_TILE + sw128_off(r, p & 7)) = v[j];
        }
      }
      fence_async_smem();  // the tensor core reads the tiles through the async proxy
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.x_ready);
    }
    const int grp = (warp - W_DQ0) >> 2;
    const int q = warp & 3;       // tensor-memory lane quarter of this warp
    const int o = q * 32 + lane;  // weight row = tensor-memory lane
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    int total = L.nA;
    bool planned = false;
    for (int i = grp; !__any_sync(0xFFFFFFFFu, *abort); i += 2) {  // warp-uniform exit
      if (i >= total && !planned) {
        total = __shfl_sync(0xFFFFFFFFu, await_plan(), 0);
        planned = true;
      }
      if (i >= total) break;
      const Item it = item_unpack(S.items[i]);
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
        // weights times 2^-24 (subnormal form); the drains multiply it out
        dequant_packed_sub<8>(wd, __halves2bfloat162(sv, sv), __halves2bfloat162(bv, bv), r);
        tmem_st<32>(lane_base + as * 64 + m * 32, r);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.a_full[as]);
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
            for (int j = 0; j < 8; ++j) {
              const int k0 = (m0 + j) * 256 + lane * 8;
              const bool in = m0 + j < nm && k0 < h;
              wv[j] = in ? __ldg(reinterpret_cast<const uint4*>(wrow + k0)) : make_uint4(0, 0, 0, 0);
              xv[j] = in ? __ldg(reinterpret_cast<const uint4*>(xr + k0)) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (m0 + j >= nm || (m0 + j) * 256 + lane * 8 >= h) continue;
#pragma unroll
              for (int cc = 0; cc < 8; ++cc) {
                const uint32_t ww = (&wv[j].x)[cc >> 1], xw = (&xv[j].x)[cc >> 1];
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
        const int hp = h / 8;
        for (int r = ew; r < t; r += 4) {
          float s = 0.f;
          for (int p0 = lane; p0 < hp; p0 += 32 * 8) {
            uint4 xv[8], gv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int p = p0 + 32 * j;
              xv[j] = p < hp ? __ldg(reinterpret_cast<const uint4*>(P.x + (size_t)r * h) + p) : make_uint4(0, 0, 0, 0);
              gv[j] = p < hp ? __ldg(reinterpret_cast<const uint4*>(P.s_gate) + p) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
              for (int cc = 0; cc < 4; ++cc) {
                const uint32_t xw = (&xv[j].x)[cc], gw = (&gv[j].x)[cc];
                s = fmaf(bf16lo(xw), bf16lo(gw), s);
                s = fmaf(bf16hi(xw), bf16hi(gw), s);
              }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
          if (lane == 0) P.gate_vals[r] = 1.f / (1.f + __expf(-s));
        }
      }
      const size_t n_gu4 = (size_t)(t + t * k) * 2 * P.imax / 4, n_acc4 = (size_t)t * h / 4;
      const size_t n_ft = (size_t)P.max_slots * (P.imax / 128), n_h = (size_t)h / 128;
      const size_t gt = (size_t)b * 128 + etid, gs = (size_t)G * 128;
      const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
      for (size_t i = gt; i < n_gu4; i += gs) reinterpret_cast<float4*>(P.gu)[i] = z4;
      for (size_t i = gt; i < n_acc4; i += gs) reinterpret_cast<float4*>(P.acc)[i] = z4;
      for (size_t i = gt; i < n_ft; i += gs) P.ftcount[i] = 0u;
      for (size_t i = gt; i < (size_t)P.max_slots; i += gs) P.hgready[i] = 0u;
      for (size_t i = gt; i < n_h; i += gs) P.hcount[i] = 0u;
    }
    // grid-wide barrier: every call advances the counter by G, so the target
    // is the next multiple of G above this CTA's arrival
    __threadfence();
    bool ok = esync();
    uint32_t bar_target = 0;
    if (ok && etid == 0) {
      const uint32_t arrival = atomicAdd(&P.st->fused_bar, 1u);
      // (one arrival more under the MOE_STALL_GRID_BARRIER test hook: the wait runs out)
      bar_target = (arrival / (uint32_t)G + 1u) * (uint32_t)G + ((P.st->stall & MOE_STALL_GRID_BARRIER) ? 1u : 0u);
    }

    // 2. selection (rows over the four warps), grouping in one warp and the
    // rest of the list (every CTA; E <= 256, t * k <= 128).  The code runs
    // twice: a first pass on made-up logits while the other CTAs reach the
    // barrier, which writes only this CTA's scratch, then the real pass.
    // Run once per launch, this code is otherwise fetched cold, and on this
    // part the fetches more than doubled its time on the path to the first
    // routed weight copy.
    const int npairs = t * k;
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
      const bool dry = pass == 0;
      if (!dry) {
        if (ok && etid == 0 && !spin_until(&P.st->fused_bar, bar_target, abort)) df_timeout(P.st, abort, 77);
        ok = esync() && !*abort;
      }
    if (ok) {
      // rows ew and ew + 4 (t <= 8): both rows' logits in flight together
      uint64_t key0[NQ], key1[NQ];
      const int r0 = ew, r1 = ew + 4;
#pragma unroll
      for (int qq = 0; qq < NQ; ++qq) {
        const int e = lane + 32 * qq;
        const float l0 = dry ? (float)((e * 37 + r0) % 11) : __ldcg(P.logits + (size_t)r0 * P.Ep + e);
        const float l1 = dry ? (float)((e * 37 + r1) % 11) : __ldcg(P.logits + (size_t)r1 * P.Ep + e);
        key0[qq] = e < E && r0 < t ? topk_key(l0, e) : 0ull;
        key1[qq] = e < E && r1 < t ? topk_key(l1, e) : 0ull;
      }
      if (r0 < t) warp_topk_softmax<NQ>(key0, k, lane, S.idx + r0 * k, S.w + r0 * k);
      if (r1 < t) warp_topk_softmax<NQ>(key1, k, lane, S.idx + r1 * k, S.w + r1 * k);
      ok = esync();
    }
    if (ok && ew == 0) {
      for (int e = lane; e < E; e += 32) S.cnt[e] = 0;
      __syncwarp();
      for (int p = lane; p < npairs; p += 32) atomicAdd(&S.cnt[S.idx[p]], 1);
      __syncwarp();
      // lane l owns experts [l * epl, l * epl + epl): list offsets and the
      // slot of every touched expert, by a scan over the lanes
      const int epl = (E + 31) / 32, e0 = lane * epl;
      int sn = 0, su = 0;
      for (int j = 0; j < epl; ++j) {
        const int e = e0 + j;
        const int c = e < E ? S.cnt[e] : 0;
        sn += c, su += c > 0;
      }
      int in = sn, iu = su;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int yn = __shfl_up_sync(0xFFFFFFFFu, in, o), yu = __shfl_up_sync(0xFFFFFFFFu, iu, o);
        if (lane >= o) in += yn, iu += yu;
      }
      int pos = in - sn, slot = iu - su;
      for (int j = 0; j < epl; ++j) {
        const int e = e0 + j;
        if (e >= E) break;
        const int c = S.cnt[e];
        S.off[e] = pos;
        if (c > 0) {
          ++slot;
          S.slot_e[slot] = e, S.slot_row0[slot] = pos, S.slot_n[slot] = c;
        }
        pos += c;
        S.cnt[e] = 0;  // from here: rows placed per expert
      }
      if (lane == 31) S.off[E] = in, S.n_touched = iu;
      if (lane == 0) S.slot_n[0] = t;
      __syncwarp();
      // stable placement, row by row (a row names an expert once, so the
      // lanes of one row touch distinct experts)
      for (int r = 0; r < t; ++r) {
        if (lane < k) {
          const int p = r * k + lane, e = S.idx[p];
          const int at = S.off[e] + S.cnt[e];
          S.cnt[e] += 1;
          S.rows[at] = r;
          S.wts[at] = S.w[p];
          if (b == 0 && !dry) P.csr.slot_of[p] = at;
        }
        __syncwarp();
      }
    }
    if (ok) ok = esync();
    if (ok) {
      // the rest of the list
      const int n = S.n_touched;
      const int rg = n * L.per_gu, rd = n * L.per_dn;
      L.rb0 = split(rg, b, G), L.nB = split(rg, b + 1, G) - L.rb0;
      L.rd0 = split(rd, b, G), L.nD = split(rd, b + 1, G) - L.rd0;
      // (the first pass writes entries past part A, which no role reads
      // before `ready`, and leaves n_items alone)
      const int total = L.total();
      if (total > D_MAX_ITEMS) {  // excluded by decode_fused_ok
        if (etid == 0 && !dry) df_timeout(P.st, abort, 68);
        ok = dry;
      } else {
        for (int i = L.nA + etid; i < total; i += 128) S.items[i] = L.entry(i);
        if (etid == 0 && !dry) S.n_items = total;
      }
      for (int i = etid; i < L.nht; i += 128) S.htcnt[i] = 0;
      if (b == 0 && !dry) {
        for (int p = etid; p < npairs; p += 128) {
          P.idx[p] = S.idx[p];
          P.w[p] = S.w[p];
          P.csr.rows[p] = S.rows[p];
          P.csr.weights[p] = S.wts[p];
        }
        for (int e = etid; e <= E; e += 128) P.csr.offsets[e] = S.off[e];
      }
      ok = esync() && ok;
    }
    }
    // parts B, C, D are known: release the other roles (an abort releases
    // them too; they read the flag)
    if (etid == 0) mbar_arrive(&S.ready);

    // 3. epilogue: drain the segments in list order
    const int qd = warp & 3;  // tensor-memory lane quarter of this warp
    const uint32_t lane_base = tmem + ((uint32_t)(qd * 32) << 16);
    const int total = ok ? S.n_items : 0;
    uint32_t u = 0;
    int seg_n = 0;
    for (int i = 0; ok && i < total; ++i) {
      const Item it = item_unpack(S.items[i]);
      ++seg_n;
      if (!it.closes) continue;
      const int ab = (int)(u % D_NACC);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&S.acc_full[ab], (u / D_NACC) & 1, abort, D_WAIT_NS))) {
        if (lane == 0) df_timeout(P.st, abort, 78);
        ok = false;
        break;
      }
      tc_fence_after();
      const int n_tok = S.slot_n[it.slot];
      const int row0 = it.slot == 0 ? -1 : S.slot_row0[it.slot];
      if (it.gu) {
        uint32_t gv[16], uv[16];
        tmem_ld16(lane_base + D_ACC_COL + ab * 32, gv);
        tmem_ld16(lane_base + D_ACC_COL + ab * 32 + 16, uv);
        tmem_ld_wait();
        tmem_ld_fence(gv);
        tmem_ld_fence(uv);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.acc_empty[ab]);
        // column j of the accumulator is x row j; keep the slot's rows
        const int f = it.tile * 128 + qd * 32 + lane;
        float* gb = P.gu + (size_t)(row0 < 0 ? 0 : t + row0) * 2 * P.imax;  // [row][gate, up][feature]
        for (int n = 0; n < n_tok; ++n) {
          const int r = row0 < 0 ? n : S.rows[row0 + n];
          float gval = 0.f, uval = 0.f;
#pragma unroll
          for (int j = 0; j < D_MAX_T; ++j)
            if (j == r) gval = __uint_as_float(gv[j]), uval = __uint_as_float(uv[j]);
          atomicAdd(gb + (size_t)(2 * n) * P.imax + f, gval * 0x1p24f);  // the weights' 2^-24 out (exact)
          atomicAdd(gb + (size_t)(2 * n + 1) * P.imax + f, uval * 0x1p24f);
        }
        __threadfence();
        if (!esync()) {
          ok = false;
          break;
        }
        const size_t ft = (size_t)it.slot * (P.imax / 128) + it.tile;
        if (etid == 0) {
          const uint32_t before = atomicAdd(&P.ftcount[ft], (uint32_t)seg_n);
          S.last = before + (uint32_t)seg_n == (uint32_t)L.nkc;
          __threadfence();
        }
        if (!esync()) {
          ok = false;
          break;
        }
        if (S.last) {
          // this CTA completed the feature tile: silu(gate) * up of its 128
          // features for the slot's rows, as the two B tiles of the down pass
          for (int qq = etid; qq < 2 * 16 * 8; qq += 128) {
            const int c = qq >> 7, n = (qq >> 3) & 15, pc = qq & 7;
            uint32_t pk[4] = {0u, 0u, 0u, 0u};
            if (n < n_tok) {
#pragma unroll
              for (int e2 = 0; e2 < 4; ++e2) {
                const int fj = it.tile * 128 + c * 64 + pc * 8 + 2 * e2;
                const float* gr = gb + (size_t)(2 * n) * P.imax + fj;
                const float2 g2 = __ldcg(reinterpret_cast<const float2*>(gr));
                const float2 u2 = __ldcg(reinterpret_cast<const float2*>(gr + P.imax));
                const float v0 = silu_mul_fast(g2.x, u2.x), v1 = silu_mul_fast(g2.y, u2.y);
                pk[e2] = ((uint32_t)f2bf(v1) << 16) | f2bf(v0);
              }
            }
            uint8_t* tile = P.hg + ((size_t)it.slot * (P.imax / D_KC) + it.tile * 2 + c) * D_TILE;
            *reinterpret_cast<uint4*>(tile + sw128_off(n, pc)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
          fence_async_global();  // bulk copies read the tiles
          __threadfence();
          if (!esync()) {
            ok = false;
            break;
          }
          if (etid == 0) atomicAdd(P.hgready + it.slot, 1u);
        }
      } else {
        uint32_t yv[16];
        tmem_ld16(lane_base + D_ACC_COL + ab * 32, yv);
        tmem_ld_wait();
        tmem_ld_fence(yv);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.acc_empty[ab]);
        // column n is the slot's n-th row: weight * y into the block accumulator
        const int col = it.tile * 128 + qd * 32 + lane;
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
            atomicAdd(P.acc + (size_t)r * h + col, (wt * 0x1p24f) * __uint_as_float(yv[n]));  // 2^-24 out
          }
        }
        if (etid == 0) S.htcnt[it.tile] += seg_n;
      }
      seg_n = 0;
      ++u;
    }

    // 4. output tiles this CTA completes (after every epilogue thread's additions)
    __threadfence();
    ok = esync() && ok && !*abort;
    if (ok) {
      const uint32_t per_tile = (uint32_t)(S.n_touched * L.nkd_r + L.nkd_s);
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

size_t cdiv(size_t a, size_t b) { return (a + b - 1) / b; }

}  // namespace

bool decode_fused_ok(const moe_dims& d, uint32_t flags) {
  if (!(d.t <= D_MAX_T && d.E <= D_MAX_E && d.h <= D_MAX_H && (flags & MOE_PACKED_WEIGHTS) &&
        (d.bits == 0 || d.bits == 4) &&
        (flags & MOE_FUSED_DECODE) &&
        !(flags & (MOE_DETERMINISTIC | MOE_FORCE_SMALL_T | MOE_FORCE_LARGE_T | MOE_SIMPLE_KERNELS))))
    return false;
  // the longest list a CTA can get must fit its table
  const size_t G = (size_t)sm_count(), nkc = d.h / D_KC, nht = d.h / 128;
  const size_t slots_r = (size_t)(d.E < d.t * d.k ? d.E : d.t * d.k);
  const size_t most = cdiv((size_t)(d.shared_inter / 128) * nkc, G) + cdiv(nht * (d.shared_inter / D_KC), G) +
                      cdiv(slots_r * (d.inter / 128) * nkc, G) + cdiv(slots_r * nht * (d.inter / D_KC), G);
  return G > 0 && most <= (size_t)D_MAX_ITEMS;
}

size_t decode_fused_ws_bytes(const moe_dims& d) {
  const int imax = d.inter > d.shared_inter ? d.inter : d.shared_inter;
  const int slots = 1 + (d.E < d.t * d.k ? d.E : d.t * d.k);
  const int Ep = (d.E + 15) / 16 * 16;
  return align_up((size_t)d.t * Ep * 4, 256) + align_up((size_t)d.t * 4, 256) +
         align_up((size_t)(d.t + d.t * d.k) * 2 * imax * 4, 256) + align_up((size_t)d.t * d.h * 4, 256) +
         align_up((size_t)slots * (imax / 128) * 4, 256) + align_up((size_t)slots * 4, 256) +
         align_up((size_t)slots * (imax / D_KC) * D_TILE, 256) + align_up((size_t)(d.h / 128) * 4, 256);
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
  P.gu = reinterpret_cast<float*>(take((size_t)(d.t + d.t * d.k) * 2 * P.imax * 4));
  P.acc = reinterpret_cast<float*>(take((size_t)d.t * d.h * 4));
  P.ftcount = reinterpret_cast<uint32_t*>(take((size_t)P.max_slots * (P.imax / 128) * 4));
  P.hgready = reinterpret_cast<uint32_t*>(take((size_t)P.max_slots * 4));
  P.hg = reinterpret_cast<uint8_t*>(take((size_t)P.max_slots * (P.imax / D_KC) * D_TILE));
  P.hcount = reinterpret_cast<uint32_t*>(take((size_t)(d.h / 128) * 4));
  P.st = st;
  const int NQ = (d.E + 31) / 32;
  if (NQ <= 1) return launch_df<1>(P, stream);
  if (NQ <= 2) return launch_df<2>(P, stream);
  if (NQ <= 4) return launch_df<4>(P, stream);
  return launch_df<8>(P, stream);
}

}  // namespace moe

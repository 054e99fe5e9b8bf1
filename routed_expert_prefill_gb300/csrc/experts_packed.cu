// Expert FFNs on pre-packed (tile-contiguous) weights: the streaming-friendly
// form of the grouped GEMMs of cherenkov qwen4_exp, prefill/experts.rs,
// pf_experts (gather_rows -> gate/up quantised matmuls -> silu_mul -> down
// quantised matmul -> scatter_add_rows, plus the shared expert).
//
// Packed weight record (moe_pack_experts), per expert (the shared expert has
// its own record with inter = shared_inter):
//   gate/up part: for each 128-row feature tile rt, for each 64-wide K chunk
//     kc: [gate block][up block], where a block is 128 rows x 32 bytes of
//     4-bit codes, then 128 bf16 scales, then 128 bf16 biases (4608 bytes).
//   down part: for each 128-row tile of h, for each 64-wide K chunk of
//     inter: one block.
//   Inside each 32-bit word of codes (8 consecutive K), even K sit in the low
//   half and odd K in the high half (K0 K2 K4 K6 | K1 K3 K5 K7, 4 bits each),
//   so (word >> 4i) & 0x000F000F is the pair (K2i, K2i+1).
// Scales and biases are rounded to bf16 once, when packing.
//
// Per call:
//   schedule: tiles of <= 128 rows per expert, largest first, each with a
//     padded-row offset (rows rounded up to 16).
//   gather:   the token rows of every tile are copied, chunk by chunk, into
//     the 128-byte-swizzled K-major image the MMA reads (xg), so one bulk
//     copy moves a whole B stage.
//   gateup:   warp 0 streams packed weight blocks (one bulk copy per stage
//     of one or two K chunks), warp 10 streams xg stages, two groups of
//     four warps take alternate stages and dequantise one weight row per
//     thread
//     (w = fma(q, s, b) in bf16) straight into TMEM with tcgen05.st, warps 1
//     and 15 issue the gate and the up tcgen05.mma streams with A in TMEM
//     and B in shared memory, and one or two four-warp epilogue groups drain
//     the gate and up accumulators into registers (silu(gate) * up), free
//     TMEM for the next unit, and write hg, again as swizzled K-major
//     images, in 16-byte pieces through per-warp staging.
//   down:     the same pipeline on the down blocks and hg images, with a
//     double-buffered accumulator; the epilogue scales by the routing weight
//     and, transposed through per-warp staging, adds 16-byte pieces into the
//     fp32 block accumulator (reductions) or, deterministic mode, stores per
//     list position.
// Every mbarrier wait is bounded (2 s of global time); a wait that gives up
// records MOE_ETIMEOUT, raises a CTA-wide abort flag, lets in-flight copies
// and MMAs land, frees TMEM and returns.
#include <type_traits>
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using namespace tc;

// Rows per tile (MMA N): 128; 64 for chunks whose experts see few rows each
// (the smaller accumulators then leave room for a deeper A ring); 160 for
// chunks whose experts see about 100 rows or more (one tile per expert
// instead of two part-empty ones, and each dequantised weight block serves
// more tokens).  160 rather than 192: the gate and up accumulators of a
// 160-row tile leave three A stages in tensor memory instead of two, and
// with two the dequantisation of stage s + 2 waited for stage s's MMAs and
// the tensor pipe idled; at t = 4096, E = 256 hardly any expert sees more
// than 160 rows.
constexpr int PTILE = 128;
constexpr int PTILE_SMALL = 64;
constexpr int PTILE_LARGE = 160;  // experts with ~100 rows or more: one tile for up to 160 rows
constexpr int KC = 64;      // K per chunk = one quantisation group
// One packed 128 x 64 block at BITS bits per code: 128 rows of 8 * BITS
// code bytes, then 128 bf16 scales and 128 bf16 biases.
__host__ __device__ constexpr int qb_bytes(int bits) { return 1024 * bits + 512; }
constexpr uint64_t WAIT_NS = 2000000000ull;

constexpr int W_CODE = 0, W_MMA = 1, W_DQ0 = 2, W_B = 10, W_EPI0 = 11, W_MMA2 = 15, W_EPI1 = 16;
// 0 code, 1 MMA (gate / down), 2-9 dequant (two groups), 10 B, 11-14
// epilogue, 15 MMA (up); launched with 20 warps, 16-19 form a second
// epilogue group that takes alternate 16-column steps.  The second group
// pays where the epilogue of a unit is long against its main loop
// (128-row tiles; for down, a short inter), and otherwise only takes issue
// slots from the dequantisation warps.
constexpr int KWARPS = 20;
static_assert(W_EPI0 + 4 == W_MMA2 && W_MMA2 + 1 == W_EPI1 && W_EPI1 + 4 == KWARPS, "warp roles");
constexpr int KTHREADS = KWARPS * 32;
constexpr int KTHREADS_1 = 16 * 32;
constexpr int SMEM_MAX = 232448;      // dynamic shared memory of one CTA (227 KB)
constexpr int CPS_DEFAULT = 2;        // K chunks per code stage and per A stage (see PCfg)

// TMEM (512 columns): NACC accumulator buffers of ACC_COLS columns (gate/up:
// gate then up, PT columns each), then the A ring of SA stages.
// CP K chunks per stage: 2, or 4 for the down pass on 64-row tiles (its
// blocks are half the gate/up stage's, so the per-stage waits and fences
// would otherwise be spread over only two blocks per warp).
// Kernel modes: the down pass on one 128-row output tile per unit, the
// gate/up pass, and the down pass on two adjacent output tiles per unit.  In
// the paired modes two weight matrices (gate and up, or two output tiles)
// share every token stage: two MMA issuers, two accumulators, one token
// image read for both, which halves the down pass's token-image ingest per
// weight block.
constexpr int MODE_DN = 0, MODE_GU = 1, MODE_DN2 = 2;

template <int MODE, int PT, int CP, int BITS>
struct PCfg {
  static constexpr int QB = qb_bytes(BITS);               // bytes of one packed block
  static constexpr int ROWB = 8 * BITS;                   // code bytes of one row of a block
  static constexpr bool GATEUP = MODE == MODE_GU;
  static constexpr bool PAIRED = MODE != MODE_DN;
  static constexpr int CPS = CP;
  static constexpr int NMAT = PAIRED ? 2 : 1;
  static constexpr int C_STAGE = CPS * NMAT * QB;        // packed blocks of one stage (QB at BITS)
  static constexpr int A_STAGE = CPS * NMAT * 32;        // TMEM columns per A stage
  static constexpr int NACC = PAIRED ? 1 : 2;            // accumulator buffers
  static constexpr int ACC_COLS = PAIRED ? 2 * PT : PT;  // TMEM columns per accumulator buffer
  static constexpr int A_COL = NACC * ACC_COLS;          // first column of the A ring
  static constexpr int SA = (512 - A_COL) / A_STAGE;     // A stages: 2 / 4 at PT 128, 3 / 3 at PT 64, 3 / 3 at PT 160
  static constexpr int NISS = PAIRED ? 2 : 1;            // MMA issuing threads (one per matrix)
  // Token-tile stages, and the ring takes all the shared memory the code
  // ring, the epilogue staging and the barriers leave.  On 160-row tiles a
  // stage holds CP chunks of a full tile (every A stage reads a single B
  // stage) and the ring is seven stages deep: the gathered token images
  // arrive several stage times after they are requested, so the ring's
  // depth is what hides that latency.  On smaller tiles a stage is 32 or 64
  // KB and holds as many chunks as fit (fewer, larger stages measured
  // faster there).
  static constexpr int B_STAGE =
      PT > 128 ? CP * PT * 128 : (CP * PT * 128 > 32768 ? 65536 : 32768);
  static constexpr int EPI_BYTES = (GATEUP ? 1 : 8) * PT * 8 + 8 * (GATEUP ? 16 * 16 : 16 * 32) * 4;
  // Code stages (as many as leave enough token stages): twelve on gate/up and
  // eight on the paired down pass and on 64-row tiles, where the weight
  // stream is what the stages wait for (at t4096 h4096 E256 against four:
  // gate/up 618 -> 601 us with eight, 598 with twelve; paired down 405 ->
  // 387 us with eight, 403 with twelve, its token ring then too short);
  // four on the single-matrix down pass with larger tiles.
  // (on tiles over 128 rows at least five token stages stay: with wider
  // codes the code stages would otherwise leave the token ring too short)
  static constexpr int SB_MIN = PT > 128 ? 5 : 2;
  static constexpr int SC_FIT = (SMEM_MAX - 2048 - EPI_BYTES - SB_MIN * B_STAGE) / C_STAGE;
  static constexpr int SC_WANT = PT <= 64 ? 8 : GATEUP ? 12 : PAIRED ? 8 : 4;
  static constexpr int SC = SC_WANT < SC_FIT ? SC_WANT : (SC_FIT < 4 ? 4 : SC_FIT);
  static constexpr int SB_FIT = (SMEM_MAX - 1024 - SC * C_STAGE - EPI_BYTES - 1024) / B_STAGE;
  static constexpr int SB = SB_FIT > 16 ? 16 : SB_FIT;
  static constexpr int B_RING = SB * B_STAGE;
  // A-ring slots are released per stage (one empty barrier each, committed
  // by every issuer after the stage's MMAs).  Releasing them block by block,
  // so that a group could rewrite a slot while the tensor pipe still read its
  // later blocks, paid on the paired passes before their issue loops were
  // warp-uniform; since then it costs more than it gains (gate/up 592 ->
  // 584 us, paired down 385 -> 376 us without it at t4096 h4096 E256).
  // Paired down pass: each output tile's accumulator has its own full and
  // empty barriers, and the epilogue drains tile 0 first, so tile 0's
  // issuer starts the next unit while tile 1 is still drained (as far as
  // the shared A slots let it run ahead).  (Measured: giving each
  // dequantisation group one matrix of every stage instead, so that the two
  // matrices' pipelines decouple fully, was slower on both paired passes:
  // every group then pays the per-stage waits twice as often.)
  static constexpr bool ACC_SPLIT = MODE == MODE_DN2;
  static_assert(SA >= 2, "the A ring needs a stage per dequantisation group");
  static_assert(SB >= 2 && B_STAGE % 1024 == 0, "token-tile ring");
  static_assert(SB <= 32 && SC <= 32, "stage bit masks");
};

__host__ __device__ inline size_t gu_bytes(int h, int I, int bits = 4) {
  return (size_t)(I / 128) * (h / KC) * 2 * qb_bytes(bits);
}
__host__ __device__ inline size_t rec_bytes(int h, int I, int bits = 4) {
  return gu_bytes(h, I, bits) + (size_t)(h / 128) * (I / KC) * qb_bytes(bits);
}

__device__ __forceinline__ uint32_t pack_word(uint32_t w) {
  return (w & 0xFu) | (((w >> 4) & 0xFu) << 16) | (((w >> 8) & 0xFu) << 4) | (((w >> 12) & 0xFu) << 20) |
         (((w >> 16) & 0xFu) << 8) | (((w >> 20) & 0xFu) << 24) | (((w >> 24) & 0xFu) << 12) |
         (((w >> 28) & 0xFu) << 28);
}

// 2 bits: a word of 16 codes (code m at bits 2m) becomes pairs (K2i,
// K2i+1) at (w >> 2i) & 0x00030003.
__device__ __forceinline__ uint32_t pack_word2(uint32_t w) {
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    r |= (((w >> (4 * i)) & 3u) << (2 * i)) | (((w >> (4 * i + 2)) & 3u) << (16 + 2 * i));
  return r;
}
// 8 bits: a word of 4 codes (code m at bits 8m) becomes pairs (K2i, K2i+1)
// at (w >> 8i) & 0x00FF00FF.
__device__ __forceinline__ uint32_t pack_word8(uint32_t w) { return __byte_perm(w, 0, 0x3120); }

// 3 bits: a row's 64 codes (24 source bytes, code k at bits [3k, 3k + 3))
// become two planes.  The low two bits of each code form four words in the
// 2-bit pair layout; the high bit of pair p = 8j + i (codes K 2p, K 2p + 1)
// goes to bits p % 16 (even code) and 16 + p % 16 (odd code) of word
// p / 16 of the high plane.
__device__ __forceinline__ void pack_row3(const uint32_t (&src)[6], uint32_t (&lo)[4], uint32_t (&hi)[2]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) lo[j] = 0;
  hi[0] = hi[1] = 0;
#pragma unroll
  for (int k = 0; k < 64; ++k) {
    const int bit = 3 * k, wi = bit >> 5, off = bit & 31;
    uint32_t v = src[wi] >> off;
    if (off > 29) v |= src[wi + 1] << (32 - off);
    const uint32_t q = v & 7u;
    const int pr = k >> 1, j = pr >> 3, i = pr & 7, half = (k & 1) * 16;
    lo[j] |= (q & 3u) << (half + 2 * i);
    hi[pr >> 4] |= (q >> 2) << (half + (pr & 15));
  }
}

// ----------------------------------------------------------------------------
// Packing: one 128-thread block per packed block (thread = weight row).
// Source records hold BITS-bit codes, each row least significant bit first.
// ----------------------------------------------------------------------------
template <int BITS>
__global__ void __launch_bounds__(128)
pack_kernel(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales,
            const uint16_t* __restrict__ biases, int h, int I, size_t src_rec_bytes, size_t src_rec_groups,
            uint8_t* __restrict__ dst) {
  constexpr int QBB = qb_bytes(BITS), ROWB = 8 * BITS;  // block bytes; code bytes of a row's 64 K
  pdl_wait();
  pdl_trigger();
  const int rec = blockIdx.y;
  const int nkc_gu = h / KC, nkc_d = I / KC;
  const int nblk_gu = (I / 128) * nkc_gu;  // gate/up block pairs
  int blk = blockIdx.x;
  int mat, rt, kc, K, rows;
  size_t dst_off;
  if (blk < 2 * nblk_gu) {
    const int pair = blk >> 1;
    mat = blk & 1;  // 0 gate, 1 up
    rt = pair / nkc_gu;
    kc = pair % nkc_gu;
    K = h;
    rows = I;
    dst_off = (size_t)pair * 2 * QBB + (size_t)mat * QBB;
  } else {
    blk -= 2 * nblk_gu;
    mat = 2;
    rt = blk / nkc_d;
    kc = blk % nkc_d;
    K = I;
    rows = h;
    dst_off = gu_bytes(h, I, BITS) + (size_t)blk * QBB;
  }
  const int o = threadIdx.x;
  const size_t mat_bytes = (size_t)I * h * BITS / 8, mat_groups = (size_t)I * h / KC;
  const uint8_t* src =
      codes + rec * src_rec_bytes + mat * mat_bytes + (size_t)(rt * 128 + o) * (K * BITS / 8) + kc * ROWB;
  const size_t g = rec * src_rec_groups + mat * mat_groups + (size_t)(rt * 128 + o) * (K / KC) + kc;
  uint8_t* d = dst + rec * rec_bytes(h, I, BITS) + dst_off;
  if constexpr (BITS == 3) {
    uint32_t w[6], lo[4], hi[2];
#pragma unroll
    for (int v = 0; v < 3; ++v) {
      const uint2 c = reinterpret_cast<const uint2*>(src)[v];
      w[2 * v] = c.x, w[2 * v + 1] = c.y;
    }
    pack_row3(w, lo, hi);
    uint2* dr = reinterpret_cast<uint2*>(d + o * ROWB);
    dr[0] = make_uint2(lo[0], lo[1]);
    dr[1] = make_uint2(lo[2], lo[3]);
    dr[2] = make_uint2(hi[0], hi[1]);
  } else {
#pragma unroll
    for (int v = 0; v < ROWB / 16; ++v) {
      uint4 c = reinterpret_cast<const uint4*>(src)[v];
      if (BITS == 2) c.x = pack_word2(c.x), c.y = pack_word2(c.y), c.z = pack_word2(c.z), c.w = pack_word2(c.w);
      if (BITS == 4) c.x = pack_word(c.x), c.y = pack_word(c.y), c.z = pack_word(c.z), c.w = pack_word(c.w);
      if (BITS == 8) c.x = pack_word8(c.x), c.y = pack_word8(c.y), c.z = pack_word8(c.z), c.w = pack_word8(c.w);
      reinterpret_cast<uint4*>(d + o * ROWB)[v] = c;
    }
  }
  __nv_bfloat16 sb = h2bf(scales[g]), bb = h2bf(biases[g]);
  reinterpret_cast<__nv_bfloat16*>(d + 128 * ROWB)[o] = sb;
  reinterpret_cast<__nv_bfloat16*>(d + 128 * ROWB + 256)[o] = bb;
  (void)rows;
}

// ----------------------------------------------------------------------------
// Gather: token rows of every tile -> swizzled K-major images.  Grid
// (tile, group of 8 rows); one warp copies one row.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
gather_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ rows, const SchedHdr* hdr,
              const int4* __restrict__ tiles, int t, int h, int E, uint16_t* __restrict__ xg, DeviceStatus* st) {
  pdl_wait();
  pdl_trigger();
  if ((int)blockIdx.x >= hdr->n_tiles) return;
  const int4 T = tiles[blockIdx.x];
  const int n = T.z, Nm = (n + 15) & ~15;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = blockIdx.y * 8 + warp;
  // rows n .. Nm-1 pad the tile to the MMA's 16-column granule: they feed
  // only accumulator columns that the epilogues drop, so they are left as
  // they are (a one-row decode tile copies one row, not sixteen)
  if (j >= n) return;
  uint8_t* base = reinterpret_cast<uint8_t*>(xg + (size_t)T.w * h);
  const int npieces = h / 8;
  const int r = (T.x == E) ? T.y + j : rows[T.y + j];
  const bool ok = (r >= 0 && r < t);
  if (!ok && lane == 0) raise_flag(st, FLAG_BAD_ROW);
  for (int pc = lane; pc < npieces; pc += 32) {
    const uint4 v = ok ? reinterpret_cast<const uint4*>(x + (size_t)r * h)[pc] : make_uint4(0, 0, 0, 0);
    const int kc = pc >> 3, c = pc & 7;
    *reinterpret_cast<uint4*>(base + (size_t)kc * Nm * 128 + sw128_off(j, c)) = v;
  }
}

__device__ __forceinline__ void note_timeout(DeviceStatus* st, volatile int* abort, uint32_t site) {
  if (atomicOr(&st->flags, FLAG_TIMEOUT) == 0) st->timeout_site = site;
  *abort = 1;
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const int never = 0;
  mbar_wait(bar, parity, &never, 100000000ull);
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Down epilogue for 16 accumulator columns of one warp (lane = feature):
// column j goes to row s_row[j] (-1: none) of the destination, scaled by
// s_w[j].  The scaled values pass through stg ([16][32] floats) so that lane
// l then owns features 4 (l % 8) .. +3 of column 4 it + l / 8; dq points at
// this lane's first feature in destination row 0.  Plain 16-byte stores in
// deterministic mode (every destination written once), fp32 reductions
// otherwise.  The column weights w4 and this lane's destination rows rr are
// loaded by the caller before it waits for the accumulator load, and the
// four staged vectors are read before the first reduction is issued, so the
// shared-memory latencies overlap instead of adding up.
template <bool DET>
__device__ __forceinline__ void down_cols16(const uint32_t (&y)[16], const float4 (&w4)[4], const int (&rr)[4],
                                            float* stg, float* dq, int lane, int h) {
  __syncwarp();  // the previous batch's reads of stg are done
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    stg[(4 * jj + 0) * 32 + lane] = w4[jj].x * __uint_as_float(y[4 * jj + 0]);
    stg[(4 * jj + 1) * 32 + lane] = w4[jj].y * __uint_as_float(y[4 * jj + 1]);
    stg[(4 * jj + 2) * 32 + lane] = w4[jj].z * __uint_as_float(y[4 * jj + 2]);
    stg[(4 * jj + 3) * 32 + lane] = w4[jj].w * __uint_as_float(y[4 * jj + 3]);
  }
  __syncwarp();
  float4 v[4];
#pragma unroll
  for (int it = 0; it < 4; ++it) v[it] = reinterpret_cast<const float4*>(stg + (it * 4 + (lane >> 3)) * 32)[lane & 7];
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    if (rr[it] >= 0) {
      float4* d = reinterpret_cast<float4*>(dq + (size_t)(uint32_t)rr[it] * (uint32_t)h);
      if (DET) *d = v[it];
      else atomicAdd(d, v[it]);
    }
  }
}

// Dequantise one row of a packed block (64 K) into 32 bf16 pairs in K order.
// The in-word layouts are those of pack_kernel.  Every width uses the
// subnormal form of dequant_packed_sub: the code's bits read as a bf16
// number of value r * 2^-133 times s * 2^109, plus b * 2^-24, rounded once,
// which is (q s + b) * 2^-24; a code masked 2, 4 or 6 bits up reads as 4 q,
// 16 q or 64 q and takes the scale divided by that.  The accumulators then
// carry the factor 2^-24, which the epilogues multiply out (exact).
constexpr float DQ_SCALE_UP = 0x1p109f, DQ_BIAS_DOWN = 0x1p-24f, ACC_UP = 0x1p24f;

template <int BITS>
__device__ __forceinline__ void dequant_bits(const uint32_t* w, __nv_bfloat162 s2, __nv_bfloat162 b2, uint32_t* out) {
  const __nv_bfloat162 sA = __hmul2(s2, __float2bfloat162_rn(DQ_SCALE_UP));
  const __nv_bfloat162 bb = __hmul2(b2, __float2bfloat162_rn(DQ_BIAS_DOWN));
  auto fma_raw = [&](uint32_t raw, __nv_bfloat162 sc) {
    const __nv_bfloat162 r = __hfma2(*reinterpret_cast<const __nv_bfloat162*>(&raw), sc, bb);
    return *reinterpret_cast<const uint32_t*>(&r);
  };
  if constexpr (BITS == 4) {
    // word j: pairs (K 8j + 2i, K 8j + 2i + 1) at (w >> 4i) & 0x000F000F
    dequant_packed_sub<8>(w, s2, b2, out);
  } else if constexpr (BITS == 2) {
    // word j: pairs (K 16j + 2i, K 16j + 2i + 1) at (w >> 2i) & 0x00030003
    __nv_bfloat162 sc[4];
    sc[0] = sA;
#pragma unroll
    for (int i = 1; i < 4; ++i) sc[i] = __hmul2(sc[i - 1], __float2bfloat162_rn(0.25f));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t lo = w[j], hi = w[j] >> 8;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        out[8 * j + i] = fma_raw(lo & (0x00030003u << (2 * i)), sc[i]);
        out[8 * j + 4 + i] = fma_raw(hi & (0x00030003u << (2 * i)), sc[i]);
      }
    }
  } else if constexpr (BITS == 3) {
    // w[0..3]: the low two bits in the 2-bit pair layout; w[4..5]: the high
    // bits, pair p = 8j + i at bit p % 16 of each half of word 4 + p / 16.
    // The code is assembled at bits 0-2 of each half.
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int hs = 8 * (j & 1) + i;  // the high bit's position in its half
        const uint32_t hw = w[4 + (j >> 1)];
        const uint32_t hb = (hs >= 2 ? hw >> (hs - 2) : hw << (2 - hs)) & 0x00040004u;
        out[8 * j + i] = fma_raw(((w[j] >> (2 * i)) & 0x00030003u) | hb, sA);
      }
  } else {
    static_assert(BITS == 8, "2, 3, 4 or 8 bits");
    // word j: pairs (K 4j + 2i, K 4j + 2i + 1) at (w >> 8i) & 0x00FF00FF
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      out[2 * j + 0] = fma_raw(w[j] & 0x00FF00FFu, sA);
      out[2 * j + 1] = fma_raw((w[j] >> 8) & 0x00FF00FFu, sA);
    }
  }
}

// silu(g) * u of accumulators carrying the factor 2^-24 of dequant_bits: the
// same arithmetic as silu_mul_fast on (2^24 G, 2^24 U), with the powers of
// two folded into its constants (bit-identical while G U stays normal).
__device__ __forceinline__ float silu_mul_acc(float G, float U) {
  float th;
  asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(0x1p23f * G));
  return G * U * fmaf(0x1p47f, th, 0x1p47f);
}

struct PUnit {
  int e, start, n, Nm, f0, nkc, kps, pad;
  bool shared;
};

template <int MODE, int CPS, int B_STAGE>
__device__ __forceinline__ PUnit decode_punit(const TcParams& p, int u) {
  constexpr bool GATEUP = MODE == MODE_GU;
  PUnit U;
  int4 T;
  if (GATEUP) {
    const int code = p.units_gu[u];
    T = p.tiles[code >> 8];
    U.f0 = (code & 255) * 128;
  } else {
    constexpr int W = MODE == MODE_DN2 ? 256 : 128;  // output features of one unit
    const int nmt = p.h / W;
    T = p.tiles[u / nmt];
    U.f0 = (u % nmt) * W;
  }
  U.e = T.x;
  U.start = T.y;
  U.n = T.z;
  U.Nm = (T.z + 15) & ~15;
  U.pad = T.w;
  U.shared = (T.x == p.E);
  U.nkc = GATEUP ? p.h / KC : (U.shared ? p.Is : p.I) / KC;
  // K chunks per B stage: a whole number of A stages, so that every A stage
  // reads a single B stage
  U.kps = min(B_STAGE / (U.Nm * 128), U.nkc) / CPS * CPS;
  return U;
}

struct PParams {
  TcParams p;
  const uint8_t* packed;    // routed records
  const uint8_t* s_packed;  // shared record
  // Record slots (streamed records): when non-null, expert e's record is
  // record rec_map[e] of `packed`, which holds n_rec records.
  const int32_t* rec_map;
  int n_rec;
  const uint16_t* xg;       // gathered token images
  int kmax;                 // max(I, Is): hg row pitch in the padded space
};

// Record index of routed expert e: e itself, or its slot in the streamed
// layout (a slot outside [0, n_rec) is flagged and read as slot 0).
__device__ __forceinline__ int record_of(const PParams& P, int e) {
  if (!P.rec_map) return e;
  const int r = P.rec_map[e];
  if (r < 0 || r >= P.n_rec) {
    raise_flag(P.p.status, FLAG_BAD_OFFSETS);
    return 0;
  }
  return r;
}

template <int MODE, int PT, int CP, int BITS>
struct PSmem {
  static constexpr bool GATEUP = MODE == MODE_GU;
  // down epilogue: per epilogue warp, the destination row (-1: skip) and
  // weight of every column of the current tile
  alignas(16) int col_row[GATEUP ? 1 : 8][PT];
  alignas(16) float col_w[GATEUP ? 1 : 8][PT];
  // epilogue: per epilogue warp, 16 columns x its 32 features (bf16 hg for
  // gate/up, fp32 for down), the transpose that turns one value per lane
  // into 16 bytes of consecutive features
  alignas(16) float stage[8][GATEUP ? 16 * 16 : 16 * 32];
  using C = PCfg<MODE, PT, CP, BITS>;
  uint64_t code_full[C::SC], code_empty[C::SC];
  uint64_t a_full[C::SA];
  uint64_t a_empty[C::SA];
  uint64_t b_full[C::SB], b_empty[C::SB];
  uint64_t acc_full[2], acc_empty[2];  // per buffer, or per matrix (ACC_SPLIT)
  uint64_t drain[2];
  uint32_t tmem_slot;
  int abort;
};

template <int MODE, int PT, int CP, int BITS>
constexpr size_t psmem_bytes() {
  using C = PCfg<MODE, PT, CP, BITS>;
  return 1024 + (size_t)C::B_RING + (size_t)C::SC * C::C_STAGE + sizeof(PSmem<MODE, PT, CP, BITS>);
}

// This warp has issued its last load of an accumulator buffer: hand it back
// to the MMA issuer.
__device__ __forceinline__ void release_acc(uint64_t* bar, int lane) {
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

template <int MODE, int PT, int CP, int BITS>
__global__ void __launch_bounds__(KTHREADS, 1) packed_gemm_kernel(PParams P) {
  pdl_wait();
  pdl_trigger();
  using C = PCfg<MODE, PT, CP, BITS>;
  constexpr int QB = C::QB;
  constexpr bool GATEUP = C::GATEUP, PAIRED = C::PAIRED;
  constexpr int CPS = CP;
  constexpr int SB = C::SB, B_STAGE = C::B_STAGE;
  const TcParams& p = P.p;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* b_s = base;
  uint8_t* c_s = b_s + C::B_RING;
  PSmem<MODE, PT, CP, BITS>& S = *reinterpret_cast<PSmem<MODE, PT, CP, BITS>*>(c_s + C::SC * C::C_STAGE);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = p.h;
  const int egroups = blockDim.x > KTHREADS_1 ? 2 : 1;  // epilogue warpgroups
  const int unit0 = blockIdx.x, ustride = gridDim.x;

  if (GATEUP && p.zero_acc) {
    float4* acc4 = reinterpret_cast<float4*>(p.acc);
    const size_t n4 = (size_t)p.t * h / 4;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x)
      acc4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::SC; ++i) {
      mbar_init(&S.code_full[i], 1);
      mbar_init(&S.code_empty[i], 4);
    }
    for (int i = 0; i < C::SA; ++i) {
      mbar_init(&S.a_full[i], 4);
      mbar_init(&S.a_empty[i], C::NISS);
    }
    for (int i = 0; i < SB; ++i) {
      mbar_init(&S.b_full[i], 1);
      mbar_init(&S.b_empty[i], C::NISS);
    }
    for (int i = 0; i < (C::ACC_SPLIT ? 2 : C::NACC); ++i) {
      mbar_init(&S.acc_full[i], C::ACC_SPLIT ? 1 : C::NISS);
      mbar_init(&S.acc_empty[i], 4 * egroups);
    }
    mbar_init(&S.drain[0], 1);
    mbar_init(&S.drain[1], 1);
    S.abort = 0;
    fence_mbar_init();
  }
  if (warp == W_MMA) tmem_alloc(&S.tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_slot;
  volatile int* abort = &S.abort;
  const int n_units =
      GATEUP ? p.hdr->n_units_gu : (MODE == MODE_DN2 ? p.hdr->n_units_dn / 2 : p.hdr->n_units_dn);

  if (warp == W_CODE) {
    // ------------------------------------------------------------ packed weight blocks, CPS chunks per copy
    // (none under the MOE_STALL_WEIGHT_COPIES test hook: the consumers' waits run out).
    // Like the MMA issuers, the producers walk their loops as a whole warp
    // and one elected lane issues the copies.
    if (!(p.status && (p.status->stall & MOE_STALL_WEIGHT_COPIES))) {
      uint32_t it = 0;
      // stages with a copy issued, and the phase parity each was armed for
      // (bit masks: a per-thread array indexed by the stage would live in
      // local memory)
      uint32_t armed = 0, par = 0;
      bool stop = false;
      // The weight blocks of unit u: nst stages of C_STAGE bytes from the
      // returned address (paired down: blocks of the second output tile
      // `m2` bytes further on, copied block by block into [chunk][tile]).
      size_t m2 = 0;
      auto unit_codes = [&](int u, int& nst) -> const uint8_t* {
        const PUnit U = decode_punit<MODE, CP, C::B_STAGE>(p, u);
        const int Iu = U.shared ? p.Is : p.I;
        const uint8_t* rec = U.shared ? P.s_packed : P.packed + (size_t)record_of(P, U.e) * rec_bytes(h, p.I, BITS);
        nst = U.nkc / CPS;
        m2 = (size_t)(Iu / KC) * QB;
        if (GATEUP) return rec + (size_t)(U.f0 / 128) * (h / KC) * 2 * QB;
        return rec + gu_bytes(h, Iu, BITS) + (size_t)(U.f0 / 128) * (Iu / KC) * QB;
      };
      for (int u = unit0; u < n_units && !stop; u += ustride) {
        int nst;
        const uint8_t* src = unit_codes(u, nst);
        for (int st = 0; st < nst; ++st, ++it) {
          const int sc = it % C::SC;
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(&S.code_empty[sc], ((it / C::SC) & 1) ^ 1, abort, WAIT_NS))) {
            if (lane == 0) note_timeout(p.status, abort, GATEUP ? 31 : 41);
            stop = true;
            break;
          }
          if (elect_one()) {
            mbar_arrive_expect_tx(&S.code_full[sc], C::C_STAGE);
            if constexpr (MODE == MODE_DN2) {
#pragma unroll
              for (int c = 0; c < CPS; ++c)
#pragma unroll
                for (int m = 0; m < 2; ++m)
                  bulk_load(c_s + sc * C::C_STAGE + (c * 2 + m) * QB, src + m * m2 + (size_t)(st * CPS + c) * QB, QB,
                            &S.code_full[sc]);
            } else {
              bulk_load(c_s + sc * C::C_STAGE, src + (size_t)st * C::C_STAGE, C::C_STAGE, &S.code_full[sc]);
            }
          }
          __syncwarp();
          armed |= 1u << sc;
          par = (par & ~(1u << sc)) | (((it / C::SC) & 1u) << sc);
        }
        if (__any_sync(0xFFFFFFFFu, *abort)) stop = true;
      }
      if (__any_sync(0xFFFFFFFFu, *abort))
        for (int i = 0; i < C::SC; ++i)
          if ((armed >> i) & 1u) drain_wait(&S.code_full[i], (par >> i) & 1u);
    }
  } else if (warp == W_B) {
    // ------------------------------------------------------------ token images
    {
      uint32_t it = 0;
      uint32_t armed = 0, par = 0;  // as for the code stages
      bool stop = false;
      for (int u = unit0; u < n_units && !stop; u += ustride) {
        const PUnit U = decode_punit<MODE, CP, C::B_STAGE>(p, u);
        const uint8_t* src = GATEUP ? reinterpret_cast<const uint8_t*>(P.xg + (size_t)U.pad * h)
                                    : reinterpret_cast<const uint8_t*>(p.hg + (size_t)U.pad * P.kmax);
        for (int kc0 = 0; kc0 < U.nkc; kc0 += U.kps, ++it) {
          const int sb = it % SB;
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(&S.b_empty[sb], ((it / SB) & 1) ^ 1, abort, WAIT_NS))) {
            if (lane == 0) note_timeout(p.status, abort, GATEUP ? 32 : 42);
            stop = true;
            break;
          }
          const uint32_t bytes = (uint32_t)(min(U.kps, U.nkc - kc0) * U.Nm * 128);
          if (elect_one()) {
            mbar_arrive_expect_tx(&S.b_full[sb], bytes);
            bulk_load(b_s + sb * B_STAGE, src + (size_t)kc0 * U.Nm * 128, bytes, &S.b_full[sb]);
          }
          __syncwarp();
          armed |= 1u << sb;
          par = (par & ~(1u << sb)) | (((it / SB) & 1u) << sb);
        }
        if (__any_sync(0xFFFFFFFFu, *abort)) stop = true;
      }
      if (__any_sync(0xFFFFFFFFu, *abort))
        for (int i = 0; i < SB; ++i)
          if ((armed >> i) & 1u) drain_wait(&S.b_full[i], (par >> i) & 1u);
    }
  } else if (warp == W_MMA || warp == W_MMA2) {
    // ------------------------------------------------------------ MMA issuers (A in TMEM)
    // The issue loop is kept lean (no division, descriptors stepped
    // incrementally): one thread feeds each issue stream, so every
    // instruction between two MMAs delays the next one.  gate/up: warp W_MMA
    // issues the gate MMAs and W_MMA2 the up MMAs -- separate accumulators,
    // so the two streams are independent and each commit barrier counts
    // both; down: W_MMA alone (one accumulator, one fixed order).
    const int m = warp == W_MMA ? 0 : 1;
    // The whole warp walks the loop (its waits and bookkeeping stay
    // warp-uniform) and one elected lane issues: the same lane every time,
    // so its commits track its own MMAs.  Issued this way an MMA costs
    // about half the cycles of a lone lane-0 loop.
    if (PAIRED || warp == W_MMA) {
      // descriptor of token stage 0; stage sb's differs by its offset in
      // the start-address field (16-byte units; shared memory < 256 KB
      // keeps the field from overflowing), computed rather than looked up
      // in a per-thread table, which would live in local memory
      const uint64_t bstage0 = desc_sw128(smem_u32(b_s));
      uint32_t ast = 0, bit = 0, uit = 0;
      for (int u = unit0; u < n_units && !__any_sync(0xFFFFFFFFu, *abort); u += ustride, ++uit) {
        const PUnit U = decode_punit<MODE, CP, C::B_STAGE>(p, u);
        const uint32_t idesc = idesc_bf16(128, U.Nm);
        const uint32_t nm8 = (uint32_t)(U.Nm * 128) >> 4;  // descriptor step of one K chunk
        const int ab = uit % C::NACC;
        const int ai = C::ACC_SPLIT ? m : ab;  // accumulator barrier
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&S.acc_empty[ai], ((uit / C::NACC) & 1) ^ 1, abort, WAIT_NS))) {
          if (lane == 0) note_timeout(p.status, abort, GATEUP ? 33 : 43);
          break;
        }
        const uint32_t acc = tmem + ab * C::ACC_COLS;
        bool ok = true;
        int sub = 0;
        uint64_t bd = 0;
        for (int st = 0; st < U.nkc / CPS; ++st, ++ast) {
          const int sa = ast % C::SA;
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(&S.a_full[sa], (ast / C::SA) & 1, abort, WAIT_NS))) {
            if (lane == 0) note_timeout(p.status, abort, GATEUP ? 35 : 45);
            ok = false;
            break;
          }
          const uint32_t a_st = tmem + C::A_COL + sa * C::A_STAGE;
          const bool leader = elect_one();
          if (leader) tc_fence_after();
#pragma unroll
          for (int c = 0; c < CPS; ++c) {
            const int kc = st * CPS + c;
            const int sb = bit % SB;
            if (sub == 0) bd = bstage0 + (uint64_t)((uint32_t)(sb * B_STAGE) >> 4);  // b_full was observed by the dequant warps before a_full
            if (leader) {
#pragma unroll
              for (int kk = 0; kk < KC / 16; ++kk)
                mma_bf16_ta(acc + m * PT, a_st + (c * C::NMAT + m) * 32 + 8 * kk, bd + 2 * kk, idesc, (kc | kk) != 0);
            }
            bd += nm8;
            if (++sub == U.kps || kc == U.nkc - 1) {
              if (leader) mma_commit(&S.b_empty[sb]);
              ++bit;
              sub = 0;
            }
          }
          if (leader) mma_commit(&S.a_empty[sa]);
          __syncwarp();
        }
        if (!ok) break;
        if (elect_one()) mma_commit(&S.acc_full[ai]);
        __syncwarp();
      }
      if (__any_sync(0xFFFFFFFFu, *abort)) {
        if (elect_one()) mma_commit(&S.drain[m]);
        __syncwarp();
        drain_wait(&S.drain[m], 0);
      }
    }
  } else if (warp < W_B) {
    // ------------------------------------------------------------ dequant: two groups alternate stages
    const int grp = (warp - W_DQ0) >> 2;  // 0: warps 2-5, 1: warps 6-9
    const int q = warp & 3;               // TMEM lane quarter this warp may access
    const int o = q * 32 + lane;          // weight row (= TMEM lane)
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    uint32_t ast = 0, bbase = 0;  // global A stage; global B stage at the unit's start
    for (int u = unit0; u < n_units && !*abort; u += ustride) {
      const PUnit U = decode_punit<MODE, CP, C::B_STAGE>(p, u);
      bool ok = true;
      // the token stage of each A stage, counted without a division: a B
      // stage spans spb whole A stages
      const int spb = U.kps / CPS;
      int bsub = 0;
      uint32_t bcur = bbase;
      for (int st = 0; st < U.nkc / CPS; ++st, ++ast) {
        const bool b_first = bsub == 0;
        const uint32_t bst = bcur;
        if (++bsub == spb) bsub = 0, ++bcur;
        if ((int)(ast & 1) != grp) continue;
        const int sc = ast % C::SC, sa = ast % C::SA;
        const uint32_t a_par = ((ast / C::SA) & 1) ^ 1;
        // warp-uniform verdicts: the TMEM stores below are .sync.aligned, so
        // no lane may leave the loop alone when a wait gives up
        const bool got = mbar_wait(&S.code_full[sc], (ast / C::SC) & 1, abort, WAIT_NS) &&
                         mbar_wait(&S.a_empty[sa], a_par, abort, WAIT_NS);
        if (!__all_sync(0xFFFFFFFFu, got)) {
          if (lane == 0) note_timeout(p.status, abort, GATEUP ? 36 : 46);
          ok = false;
          break;
        }
        tc_fence_after();
        // The codes, scale and bias of block cm + 1 are loaded before block
        // cm is dequantised and stored (the tensor-memory store is a compiler
        // barrier), so their shared-memory latency overlaps the arithmetic.
        const uint8_t* stage_c = c_s + sc * C::C_STAGE;
        // a row's codes in 16-byte words (rows of 16, 32 or 64 bytes) or 8-byte words (3 bits, 24 bytes)
        using CW = std::conditional_t<C::ROWB % 16 == 0, uint4, uint2>;
        constexpr int NV = C::ROWB / (int)sizeof(CW);
        CW cw[NV];
#pragma unroll
        for (int v = 0; v < NV; ++v) cw[v] = reinterpret_cast<const CW*>(stage_c + o * C::ROWB)[v];
        __nv_bfloat16 sv = reinterpret_cast<const __nv_bfloat16*>(stage_c + 128 * C::ROWB)[o];
        __nv_bfloat16 bv = reinterpret_cast<const __nv_bfloat16*>(stage_c + 128 * C::ROWB + 256)[o];
#pragma unroll
        for (int cm = 0; cm < CPS * C::NMAT; ++cm) {
          CW nw[NV];
#pragma unroll
          for (int v = 0; v < NV; ++v) nw[v] = cw[v];
          __nv_bfloat16 ns = sv, nbv = bv;
          if (cm + 1 < CPS * C::NMAT) {
            const uint8_t* nb = stage_c + (cm + 1) * QB;
#pragma unroll
            for (int v = 0; v < NV; ++v) nw[v] = reinterpret_cast<const CW*>(nb + o * C::ROWB)[v];
            ns = reinterpret_cast<const __nv_bfloat16*>(nb + 128 * C::ROWB)[o];
            nbv = reinterpret_cast<const __nv_bfloat16*>(nb + 128 * C::ROWB + 256)[o];
          }
          uint32_t r[32];
          dequant_bits<BITS>(reinterpret_cast<const uint32_t*>(cw), __halves2bfloat162(sv, sv),
                             __halves2bfloat162(bv, bv), r);
          tmem_st<32>(lane_base + C::A_COL + sa * C::A_STAGE + cm * 32, r);
#pragma unroll
          for (int v = 0; v < NV; ++v) cw[v] = nw[v];
          sv = ns, bv = nbv;
        }
        if (!ok) {
          tmem_st_wait();
          break;
        }
        tmem_st_wait();
        tc_fence_before();
        // The MMA issuer waits on a_full only, and takes the A stages in
        // order: the B stage this A stage multiplies must have landed before
        // the a_full of the first A stage it serves completes.  Later A
        // stages of the same B stage are ordered after that observation by
        // the issuer's own earlier wait, so only the first one checks.
        if (b_first) {  // warp-uniform: every lane tests, waits only if it has not landed
          uint64_t* bf = &S.b_full[bst % SB];
          const uint32_t bpar = (bst / SB) & 1;
          if (!__all_sync(0xFFFFFFFFu, mbar_test(bf, bpar) || mbar_wait(bf, bpar, abort, WAIT_NS))) {
            if (lane == 0) note_timeout(p.status, abort, GATEUP ? 34 : 44);
            ok = false;
            break;
          }
        }
        __syncwarp();  // every lane's stores and fence are done
        if (elect_one()) {
          mbar_arrive(&S.a_full[sa]);
          mbar_arrive(&S.code_empty[sc]);
        }
      }
      if (!ok) break;
      bbase += (uint32_t)((U.nkc + U.kps - 1) / U.kps);
    }
  } else if (warp < W_MMA2 || warp >= W_EPI1) {
    // ------------------------------------------------------------ epilogue: two warpgroups
    // With two groups, warp pairs share a TMEM lane quarter and group `half`
    // takes the 16-column steps c = half, half + 2, ...  Each warp releases
    // the accumulator after its own last load (at once when it has no step).
    const int q = warp & 3;
    const int half = warp >= W_EPI1 ? 1 : 0;
    const int ew = half * 4 + q;  // epilogue warp index: staging buffer, row copy
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    uint32_t uit = 0;
    for (int u = unit0; u < n_units && !*abort; u += ustride, ++uit) {
      const PUnit U = decode_punit<MODE, CP, C::B_STAGE>(p, u);
      const int ab = uit % C::NACC;
      // down: this warp's copy of the tile's destination rows and weights.
      // Deterministic mode writes routed columns to their own list position
      // (weights applied when the slots are summed) and the shared expert
      // straight into the block accumulator.
      const bool to_list = p.deterministic && !U.shared;
      if (!GATEUP) {
        bool bad_row = false;
#pragma unroll
        for (int g = 0; g < PT / 32; ++g) {
          const int col = g * 32 + lane;
          int r = -1;
          float wv = 0.f;
          if (col < U.n) {
            if (to_list) {
              r = U.start + col;
              wv = 1.f;
            } else {
              if (U.shared) {
                r = U.start + col;
                wv = p.gate_vals ? p.gate_vals[r] : 1.f;
              } else {
                r = p.rows[U.start + col];
                wv = p.weights[U.start + col];
              }
              if (r < 0 || r >= p.t) bad_row = true, r = -1;
            }
          }
          S.col_row[ew][col] = r;
          S.col_w[ew][col] = wv * ACC_UP;  // the accumulators carry 2^-24 (dequant_bits)
        }
        if (bad_row) raise_flag(p.status, FLAG_BAD_ROW);
        __syncwarp();
      }
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&S.acc_full[ab], (uit / C::NACC) & 1, abort, WAIT_NS))) {
        if (lane == 0) note_timeout(p.status, abort, GATEUP ? 37 : 47);
        break;
      }
      tc_fence_after();
      const uint32_t acc = lane_base + ab * C::ACC_COLS;
      if (GATEUP) {
        // silu(gate) * up, 16 columns at a time, stored straight into the hg
        // image (no unit-sized register buffer, so the 16 independent silu
        // evaluations of a step overlap); the accumulator is released once
        // the last store has been issued
        // The 16 x 32 bf16 values of a step pass through this warp's staging
        // buffer, after which lane l stores the 16-byte chunk (4 (q % 2) +
        // l % 4) of image rows l / 4 and 8 + l / 4.
        uint8_t* img = reinterpret_cast<uint8_t*>(p.hg + (size_t)U.pad * P.kmax) + (size_t)(U.f0 / 64 + q / 2) * U.Nm * 128;
        __nv_bfloat16* stg = reinterpret_cast<__nv_bfloat16*>(S.stage[ew]);
        const int cc = (q & 1) * 4 + (lane & 3);
        const int nb = U.Nm / 16;
        if (half >= nb) release_acc(&S.acc_empty[ab], lane);
        for (int c = half; c < nb; c += egroups) {
          uint32_t g[16], v[16];
          tmem_ld16(acc + c * 16, g);
          tmem_ld16(acc + PT + c * 16, v);
          tmem_ld_wait();
          tmem_ld_fence(g);
          tmem_ld_fence(v);
          if (c + egroups >= nb) release_acc(&S.acc_empty[ab], lane);
          __syncwarp();  // the previous step's reads of the staging buffer are done
#pragma unroll
          for (int j = 0; j < 16; ++j)
            stg[j * 32 + lane] = __float2bfloat16_rn(
                c * 16 + j < U.n ? silu_mul_acc(__uint_as_float(g[j]), __uint_as_float(v[j])) : 0.f);
          __syncwarp();
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int j = half * 8 + (lane >> 2);
            const uint4 hv = reinterpret_cast<const uint4*>(stg + j * 32)[lane & 3];
            *reinterpret_cast<uint4*>(img + sw128_off(c * 16 + j, cc)) = hv;
          }
        }
      } else {
        // 16 columns at a time, transposed through this warp's staging
        // buffer: afterwards each lane holds four consecutive features of one
        // destination row, so the scatter-add issues 16-byte reductions (a
        // quarter of the requests of one float per lane, each four times
        // wider).  The accumulator is released after its last load.
        // Paired mode: output tile m's accumulator at columns m PT (features
        // f0 + 128 m); each tile has its own barriers (ACC_SPLIT), tile 0 is
        // drained and handed back first.
        float* dq = (to_list ? p.ybuf : p.acc) + U.f0 + q * 32 + (lane & 7) * 4;
        float* stg = S.stage[ew];
        const int nb = U.Nm / 16;
        bool fail = false;
        for (int m = 0; m < C::NMAT && !fail; ++m) {
          if (C::ACC_SPLIT && m > 0) {
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(&S.acc_full[m], uit & 1, abort, WAIT_NS))) {
              if (lane == 0) note_timeout(p.status, abort, 48);
              fail = true;
              break;
            }
            tc_fence_after();
          }
          const bool rel = C::ACC_SPLIT || m == C::NMAT - 1;  // this pass ends with a hand-back
          uint64_t* ebar = &S.acc_empty[C::ACC_SPLIT ? m : ab];
          if (rel && half >= nb) release_acc(ebar, lane);
          for (int c = half; c < nb; c += egroups) {
            uint32_t y[16];
            tmem_ld16(acc + m * PT + c * 16, y);
            float4 w4[4];
            int rr[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) w4[jj] = reinterpret_cast<const float4*>(&S.col_w[ew][c * 16])[jj];
#pragma unroll
            for (int it = 0; it < 4; ++it) rr[it] = S.col_row[ew][c * 16 + it * 4 + (lane >> 3)];
            tmem_ld_wait();
            tmem_ld_fence(y);
            if (rel && c + egroups >= nb) release_acc(ebar, lane);
            if (p.deterministic)
              down_cols16<true>(y, w4, rr, stg, dq + m * 128, lane, h);
            else
              down_cols16<false>(y, w4, rr, stg, dq + m * 128, lane, h);
          }
        }
        if (fail) break;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == W_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}


}  // namespace

size_t packed_record_bytes(int h, int I, int bits) { return rec_bytes(h, I, bits); }

// Tile-list capacity, sized for the smaller tiles.
size_t packed_max_tiles(const moe_dims& d) {
  return (size_t)d.t * d.k / PTILE_SMALL + d.E + d.t / PTILE_SMALL + 2;
}

// Upper bound of the padded row space (rows rounded up to 16 per tile).
size_t packed_pad_rows(const moe_dims& d) {
  return (size_t)d.t * d.k + d.t + 16 * packed_max_tiles(d);
}

cudaError_t launch_pack(const uint8_t* codes, const uint16_t* scales, const uint16_t* biases, int h, int I,
                        int nrec, int bits, uint8_t* dst, cudaStream_t stream) {
  const int nblk = 2 * (I / 128) * (h / KC) + (h / 128) * (I / KC);
  dim3 grid(nblk, nrec);
  const size_t src_bytes = (size_t)3 * I * h * bits / 8, src_groups = (size_t)3 * I * h / KC;
  if (bits == 2)
    MOE_LAUNCH("pack", stream,
               pack_kernel<2><<<grid, 128, 0, stream>>>(codes, scales, biases, h, I, src_bytes, src_groups, dst));
  else if (bits == 3)
    MOE_LAUNCH("pack", stream,
               pack_kernel<3><<<grid, 128, 0, stream>>>(codes, scales, biases, h, I, src_bytes, src_groups, dst));
  else if (bits == 8)
    MOE_LAUNCH("pack", stream,
               pack_kernel<8><<<grid, 128, 0, stream>>>(codes, scales, biases, h, I, src_bytes, src_groups, dst));
  else
    MOE_LAUNCH("pack", stream,
               pack_kernel<4><<<grid, 128, 0, stream>>>(codes, scales, biases, h, I, src_bytes, src_groups, dst));
  return cudaGetLastError();
}

template <int MODE, int PT, int CP, int BITS>
cudaError_t launch_packed_gemm(const PParams& P, cudaStream_t stream) {
  static_assert(psmem_bytes<MODE, PT, CP, BITS>() <= SMEM_MAX, "shared memory of one CTA");
  const bool two_epi = PT >= 128 && (MODE != MODE_DN || max(P.p.I, P.p.Is) <= 1024);
  cudaError_t err =
      set_smem_limit_once(packed_gemm_kernel<MODE, PT, CP, BITS>, (int)psmem_bytes<MODE, PT, CP, BITS>());
  if (err != cudaSuccess) return err;
  MOE_LAUNCH(MODE == MODE_GU ? "gateup_packed" : "down_packed", stream,
             (launch_k(packed_gemm_kernel<MODE, PT, CP, BITS>, sm_count(), two_epi ? KTHREADS : KTHREADS_1,
                       psmem_bytes<MODE, PT, CP, BITS>(), stream, P)));
  return cudaGetLastError();
}

// K chunks per stage: gate/up two (one on 160-row tiles, whose 320
// accumulator columns leave 192 for the A ring); down four when every inter
// is a multiple of 256 on tiles of up to 128 rows, else two.
template <int PT, int BITS>
cudaError_t launch_packed_gemms(const PParams& P, cudaStream_t stream) {
  constexpr int GU_CP = PT > 128 ? 1 : CPS_DEFAULT;
  cudaError_t err = launch_packed_gemm<MODE_GU, PT, GU_CP, BITS>(P, stream);
  if (err != cudaSuccess) return err;
  // down on tiles of 128 rows or more and an inner dimension of 512 or
  // more: two output tiles per unit (the token image is read once for both),
  // staged like gate/up.  Its accumulators then take the TMEM of the double
  // buffer, so part of each unit's drain is exposed; the halved ingest pays
  // for it from inter 768 on (t4096 skewed: 133 -> 127 us; t4096 h4096:
  // 517 -> 499 us when it was introduced).
  if constexpr (PT >= 128)
    if (P.p.h % 256 == 0 && max(P.p.I, P.p.Is) >= 512)
      return launch_packed_gemm<MODE_DN2, PT, GU_CP, BITS>(P, stream);
  if constexpr (PT <= 128 && BITS <= 4)
    if (P.p.I % 256 == 0 && P.p.Is % 256 == 0) return launch_packed_gemm<MODE_DN, PT, 4, BITS>(P, stream);
  return launch_packed_gemm<MODE_DN, PT, CPS_DEFAULT, BITS>(P, stream);
}

template <int BITS>
cudaError_t launch_packed_pt(const PParams& P, int pt, cudaStream_t stream) {
  return pt == PTILE_LARGE ? launch_packed_gemms<PTILE_LARGE, BITS>(P, stream)
         : pt == PTILE     ? launch_packed_gemms<PTILE, BITS>(P, stream)
                           : launch_packed_gemms<PTILE_SMALL, BITS>(P, stream);
}

cudaError_t launch_experts_packed(const ExpertsArgs& a, const uint8_t* packed, const uint8_t* s_packed,
                                  uint16_t* xg, bool deterministic, cudaStream_t stream, const PackedBatch* pb) {
  moe_dims d{a.t, a.h, a.I, a.E, a.k, a.Is};
  const size_t mt = packed_max_tiles(d);
  const int fmax = (a.I > a.Is ? a.I : a.Is) / 128;
  SchedHdr* hdr = reinterpret_cast<SchedHdr*>(a.sched);
  int4* tiles = reinterpret_cast<int4*>(a.sched + sizeof(SchedHdr));
  int* units = reinterpret_cast<int*>(tiles + mt);
  float* gate_vals = reinterpret_cast<float*>(units + mt * fmax);

  PParams P{};
  TcParams& p = P.p;
  p.t = a.t;
  p.h = a.h;
  p.I = a.I;
  p.Is = a.Is;
  p.E = a.E;
  p.k = a.k;
  p.deterministic = deterministic ? 1 : 0;
  p.offsets = a.offsets;
  p.rows = a.rows;
  p.weights = a.weights;
  p.gate_vals = (a.Is > 0 && a.s_gate) ? gate_vals : nullptr;
  p.acc = a.acc;
  p.hg = a.hg;
  p.hgs = a.hgs;
  p.ybuf = a.ybuf;
  p.hdr = hdr;
  p.tiles = tiles;
  p.units_gu = units;
  p.status = a.status;
  const bool first = !pb || pb->first, last = !pb || pb->last;
  // the fp32 block accumulator starts at zero (before the first batch)
  // unless deterministic mode's shared expert writes every element of it
  p.zero_acc = first && (!deterministic || a.Is == 0) ? 1 : 0;
  p.batch_of = pb ? pb->batch_of : nullptr;
  p.batch = pb ? pb->batch : 0;
  P.packed = packed;
  P.s_packed = s_packed;
  P.rec_map = pb ? pb->rec_map : nullptr;
  P.n_rec = pb ? pb->n_rec : a.E;
  P.xg = xg;
  P.kmax = a.I > a.Is ? a.I : a.Is;

  // Tile height by the rows an expert sees on average: 64 up to 40 rows (a
  // larger tile would be mostly padding, and the smaller accumulators leave
  // TMEM for a deeper A ring), 128 up to 96, else 160, so that experts of
  // 100-160 rows (the near-uniform t = 4096 chunks) take one tile each
  // instead of two half-empty ones.
  const long pairs = (long)a.t * a.k;
  const int pt = pairs <= 40L * a.E ? PTILE_SMALL : pairs <= 96L * a.E ? PTILE : PTILE_LARGE;
  cudaError_t err;
  if ((err = launch_schedule(p, hdr, tiles, units, (int)mt, pt, stream)) != cudaSuccess) return err;
  if (first && p.gate_vals &&
      (err = launch_shared_gate(a.x, a.s_gate, a.t, a.h, gate_vals, stream)) != cudaSuccess)
    return err;
  MOE_LAUNCH("gather", stream,
             launch_k(gather_kernel, dim3((unsigned)mt, pt / 8), 256, 0, stream, a.x, a.rows, hdr, tiles, a.t, a.h, a.E,
                                                                          xg, a.status));
  err = a.bits == 2   ? launch_packed_pt<2>(P, pt, stream)
        : a.bits == 3 ? launch_packed_pt<3>(P, pt, stream)
        : a.bits == 8 ? launch_packed_pt<8>(P, pt, stream)
                      : launch_packed_pt<4>(P, pt, stream);
  if (err != cudaSuccess) return err;
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  return last ? launch_finalize(a, deterministic, stream) : cudaSuccess;
}

}  // namespace moe

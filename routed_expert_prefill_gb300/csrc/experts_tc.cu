// Grouped expert GEMMs on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// The routed experts (cherenkov qwen4_exp, prefill/experts.rs, pf_experts:
// per expert gather_rows -> gate/up quantised matmuls -> silu_mul -> down
// quantised matmul -> scatter_add_rows) and the shared expert run as two
// persistent kernels over a device-built tile schedule:
//
//   schedule:  per expert, its CSR rows split into tiles of <= 256 rows
//              (the shared expert: all t rows), ordered largest first.
//   gateup_tc: unit = (tile, 128 output features).  The weights are the
//              MMA's M operand (128 rows of gate and 128 rows of up), the
//              gathered token rows its N operand (16..256), so one dequantised
//              weight tile serves every row of the tile.  A producer warp
//              streams the 4-bit code tiles with TMA and gathers the token
//              rows with TMA gather4 (four CSR rows per instruction, 128-byte
//              swizzle); eight warps dequantise codes to bf16
//              (w = fma(q, s, b) in bf16) straight into the UMMA K-major
//              swizzled layout; one thread issues tcgen05.mma into two TMEM
//              accumulators (gate, up); the same eight warps then read TMEM,
//              apply silu(gate) * up and write hg (bf16, CSR order).
//   down_tc:   unit = (tile, 128 output features of h); A = dequantised down
//              rows, B = hg rows (contiguous in CSR order, plain TMA tiles);
//              the epilogue multiplies by the routing weight and adds into
//              the fp32 block accumulator with atomics, or, deterministic
//              mode, writes the unweighted result per list position.
//
// Every mbarrier wait is bounded (2 s of global time); a wait that gives up
// records MOE_ETIMEOUT in the workspace status, raises a CTA-wide abort
// flag so every role leaves its loop, lets in-flight copies and MMAs land,
// frees TMEM and returns.
#include <string.h>

#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int TILE_MAX = 256;  // rows per tile (MMA N <= 256)
constexpr int KC = 64;         // K per chunk = one quantisation group
constexpr uint64_t WAIT_NS = 2000000000ull;


__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void note_timeout(DeviceStatus* st, volatile int* abort, uint32_t site) {
  if (atomicOr(&st->flags, FLAG_TIMEOUT) == 0) st->timeout_site = site;
  *abort = 1;
}

// After an abort: wait (bounded, ignoring the abort flag) for copies or MMAs
// already issued, so nothing lands in shared memory or TMEM after exit.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const int never = 0;
  mbar_wait(bar, parity, &never, 100000000ull);
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + expf(-g)) * u; }

// 64 codes of one weight row (two 16-byte words, low nibble = even K) ->
// 8 chunks of 8 bf16 (w = fma(q, s, b) with bf16 s, b, single rounding),
// written to the 128B-swizzled K-major tile row `row`.
__device__ __forceinline__ void dequant_row_store(const uint32_t (&wd)[8], __nv_bfloat162 s2, __nv_bfloat162 b2,
                                                  uint8_t* tile, int row, int chunk0, int nchunks) {
  const __nv_bfloat162 k128 = __floats2bfloat162_rn(128.f, 128.f);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    if (c >= nchunks) break;
    const uint32_t w = wd[c];
    // (128 + K0, 128 + K4), (128 + K1, 128 + K5), ... as bf16 pairs
    const uint32_t A = (w & 0x000F000Fu) | 0x43004300u;
    const uint32_t B = ((w >> 4) & 0x000F000Fu) | 0x43004300u;
    const uint32_t C = ((w >> 8) & 0x000F000Fu) | 0x43004300u;
    const uint32_t D = ((w >> 12) & 0x000F000Fu) | 0x43004300u;
    uint32_t pr[4];
    pr[0] = __byte_perm(A, B, 0x5410);  // K0, K1
    pr[1] = __byte_perm(C, D, 0x5410);  // K2, K3
    pr[2] = __byte_perm(A, B, 0x7632);  // K4, K5
    pr[3] = __byte_perm(C, D, 0x7632);  // K6, K7
    uint4 o;
    uint32_t* ov = &o.x;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 q = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&pr[i]), k128);
      __nv_bfloat162 v = __hfma2(q, s2, b2);
      ov[i] = *reinterpret_cast<uint32_t*>(&v);
    }
    *reinterpret_cast<uint4*>(tile + sw128_off(row, chunk0 + c)) = o;
  }
}

__device__ __forceinline__ __nv_bfloat162 bf2_from_half(uint16_t hb) {
  __nv_bfloat16 b = h2bf(hb);
  return __halves2bfloat162(b, b);
}

// ----------------------------------------------------------------------------
// Tile schedule (one block)
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
schedule_kernel(TcParams p, SchedHdr* hdr, int4* tiles, int* units_gu, int max_tiles, int tile_max) {
  pdl_wait();
  pdl_trigger();
  __shared__ int bucket_cnt[16], bucket_base[16], bucket_fill[16];
  __shared__ int n_tiles_s;
  __shared__ int scan_carry;
  __shared__ int warp_sums[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nexp = p.E + (p.Is > 0 ? 1 : 0);
  if (tid < 16) {
    bucket_cnt[tid] = 0;
    bucket_fill[tid] = 0;
  }
  __syncthreads();
  // pass 1: count tiles per size bucket (bucket = ceil(size / 16) - 1)
  for (int e = tid; e < nexp; e += blockDim.x) {
    if (p.batch_of && p.batch_of[e] != p.batch) continue;
    int n;
    if (e < p.E) {
      n = p.offsets[e + 1] - p.offsets[e];
      if (n < 0 || p.offsets[e] < 0 || p.offsets[e + 1] > p.t * p.k) {
        raise_flag(p.status, FLAG_BAD_OFFSETS);
        n = 0;
      }
    } else {
      n = p.t;
    }
    if (n == 0) continue;
    const int nt = (n + tile_max - 1) / tile_max;
    const int sz = (n + nt - 1) / nt;
    for (int i = 0; i < nt; ++i) {
      const int rows = min(sz, n - i * sz);
      if (rows <= 0) break;
      atomicAdd(&bucket_cnt[(rows + 15) / 16 - 1], 1);
    }
  }
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int b = 15; b >= 0; --b) {  // largest tiles first
      bucket_base[b] = run;
      run += bucket_cnt[b];
    }
    n_tiles_s = min(run, max_tiles);
  }
  __syncthreads();
  // pass 2: place tiles
  for (int e = tid; e < nexp; e += blockDim.x) {
    if (p.batch_of && p.batch_of[e] != p.batch) continue;
    int n, start;
    if (e < p.E) {
      n = p.offsets[e + 1] - p.offsets[e];
      start = p.offsets[e];
      if (n < 0 || start < 0 || p.offsets[e + 1] > p.t * p.k) n = 0;
    } else {
      n = p.t;
      start = 0;
    }
    if (n == 0) continue;
    const int nt = (n + tile_max - 1) / tile_max;
    const int sz = (n + nt - 1) / nt;
    for (int i = 0; i < nt; ++i) {
      const int rows = min(sz, n - i * sz);
      if (rows <= 0) break;
      const int b = (rows + 15) / 16 - 1;
      const int pos = bucket_base[b] + atomicAdd(&bucket_fill[b], 1);
      if (pos < max_tiles) tiles[pos] = make_int4(e, start + i * sz, rows, 0);
    }
  }
  __syncthreads();
  // gate/up units: tile-major, feature tiles of 128 (I/128 routed, Is/128 shared)
  const int nt_all = n_tiles_s;
  if (tid == 0) scan_carry = 0;
  __syncthreads();
  for (int base = 0; base < nt_all; base += blockDim.x) {
    const int i = base + tid;
    int f = 0;
    if (i < nt_all) f = (tiles[i].x == p.E) ? p.Is / 128 : p.I / 128;
    int incl = f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int s = warp_sums[lane];
      int si = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xFFFFFFFFu, si, o);
        if (lane >= o) si += y;
      }
      warp_sums[lane] = si - s;
    }
    __syncthreads();
    const int ub = scan_carry + warp_sums[warp] + incl - f;
    for (int ft = 0; ft < f; ++ft) units_gu[ub + ft] = (i << 8) | ft;
    __syncthreads();
    if (tid == blockDim.x - 1) scan_carry = ub + f;
    __syncthreads();
  }
  const int n_units_gu = scan_carry;
  __syncthreads();
  // padded-row offset of every tile (rows rounded up to 16)
  if (tid == 0) scan_carry = 0;
  __syncthreads();
  for (int base = 0; base < nt_all; base += blockDim.x) {
    const int i = base + tid;
    const int f = (i < nt_all) ? (tiles[i].z + 15) & ~15 : 0;
    int incl = f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int s = warp_sums[lane];
      int si = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xFFFFFFFFu, si, o);
        if (lane >= o) si += y;
      }
      warp_sums[lane] = si - s;
    }
    __syncthreads();
    const int ub = scan_carry + warp_sums[warp] + incl - f;
    if (i < nt_all) tiles[i].w = ub;
    __syncthreads();
    if (tid == blockDim.x - 1) scan_carry = ub + f;
    __syncthreads();
  }
  if (tid == 0) {
    hdr->n_tiles = nt_all;
    hdr->n_units_gu = n_units_gu;
    hdr->n_units_dn = nt_all * (p.h / 128);
    hdr->pad_rows = scan_carry;
  }
}

// Per-row shared-expert gate sigmoid(x_r . g): one warp per row.
__global__ void shared_gate_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ g, int t, int h,
                                   float* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (r >= t) return;
  float d = 0.f;
  for (int i = lane * 8; i < h; i += 256) {
    const uint4 xv = *reinterpret_cast<const uint4*>(x + (size_t)r * h + i);
    const uint4 gv = *reinterpret_cast<const uint4*>(g + i);
    const uint32_t* xa = &xv.x;
    const uint32_t* ga = &gv.x;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      d = fmaf(bf16lo(xa[c]), bf16lo(ga[c]), d);
      d = fmaf(bf16hi(xa[c]), bf16hi(ga[c]), d);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xFFFFFFFFu, d, o);
  if (lane == 0) out[r] = 1.f / (1.f + expf(-d));
}

// ----------------------------------------------------------------------------
// The grouped GEMM kernel (gate/up or down)
// ----------------------------------------------------------------------------
// Warp roles: 0 code producer (TMA), 1 MMA issuer + TMEM owner, 2..9 dequant +
// epilogue, 10 B producer (TMA gather4 of token rows, or TMA tiles of hg).
constexpr int W_CODE = 0, W_MMA = 1, W_DQ0 = 2, W_B = 10;
constexpr int KWARPS = 11;
constexpr int KTHREADS = KWARPS * 32;
constexpr int SA = 2;                 // dequantised A stages (one K-chunk each)
constexpr int SB = 3;                 // B stages, 32 KB each (KPS K-chunks)
constexpr int B_STAGE = 32768;

template <bool GATEUP>
struct Cfg {
  static constexpr int NMAT = GATEUP ? 2 : 1;         // gate + up, or down
  static constexpr int CPS = GATEUP ? 2 : 4;          // K-chunks per code stage
  static constexpr int SC = GATEUP ? 4 : 5;           // code stages
  static constexpr int C_STAGE = NMAT * 128 * CPS * 32;
  static constexpr int A_STAGE = NMAT * 128 * 128;
  static constexpr int TMEM_COLS = GATEUP ? 512 : 256;
};

template <bool GATEUP>
struct KSmem {
  uint64_t code_full[Cfg<GATEUP>::SC], code_empty[Cfg<GATEUP>::SC];
  uint64_t a_full[SA], a_empty[SA];
  uint64_t b_full[SB], b_empty[SB];
  uint64_t acc_full, acc_empty, drain;
  uint32_t tmem_slot;
  int abort;
  int rowidx[TILE_MAX];
};

template <bool GATEUP>
constexpr size_t kernel_smem() {
  return 1024 + (size_t)SA * Cfg<GATEUP>::A_STAGE + (size_t)SB * B_STAGE +
         (size_t)Cfg<GATEUP>::SC * Cfg<GATEUP>::C_STAGE + sizeof(KSmem<GATEUP>);
}

// What a unit is, decoded identically by every role.
struct Unit {
  int e;        // expert, E = shared
  int start;    // first CSR position (routed) or row (shared)
  int n;        // rows
  int Nm;       // MMA N = rows rounded up to 16
  int f0;       // first output feature of the unit
  int nkc;      // K-chunks
  int kps;      // K-chunks per B stage
  bool shared;
};

template <bool GATEUP>
__device__ __forceinline__ Unit decode_unit(const TcParams& p, int u) {
  Unit U;
  int4 T;
  if (GATEUP) {
    const int code = p.units_gu[u];
    T = p.tiles[code >> 8];
    U.f0 = (code & 255) * 128;
  } else {
    const int nmt = p.h / 128;
    T = p.tiles[u / nmt];
    U.f0 = (u % nmt) * 128;
  }
  U.e = T.x;
  U.start = T.y;
  U.n = T.z;
  U.Nm = (T.z + 15) & ~15;
  U.shared = (T.x == p.E);
  U.nkc = GATEUP ? p.h / KC : (U.shared ? p.Is : p.I) / KC;
  U.kps = min(TILE_MAX / U.Nm, U.nkc);
  return U;
}

template <bool GATEUP>
__global__ void __launch_bounds__(KTHREADS, 1)
expert_gemm_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_scodes,
                   const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_sb, TcParams p) {
  pdl_wait();
  pdl_trigger();
  using C = Cfg<GATEUP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint8_t* a_s = base;
  uint8_t* b_s = a_s + SA * C::A_STAGE;
  uint8_t* c_s = b_s + SB * B_STAGE;
  KSmem<GATEUP>& S = *reinterpret_cast<KSmem<GATEUP>*>(c_s + C::SC * C::C_STAGE);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = p.h;

  if (GATEUP && p.zero_acc) {
    // The fp32 block accumulator starts at zero (atomic mode, or no shared
    // expert to initialise it); the down kernel runs after this one.
    float4* acc4 = reinterpret_cast<float4*>(p.acc);
    const size_t n4 = (size_t)p.t * h / 4;
    for (size_t i = (size_t)blockIdx.x * KTHREADS + threadIdx.x; i < n4; i += (size_t)gridDim.x * KTHREADS)
      acc4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::SC; ++i) {
      mbar_init(&S.code_full[i], 1);
      mbar_init(&S.code_empty[i], 8);
    }
    for (int i = 0; i < SA; ++i) {
      mbar_init(&S.a_full[i], 8);
      mbar_init(&S.a_empty[i], 1);
    }
    for (int i = 0; i < SB; ++i) {
      mbar_init(&S.b_full[i], 1);
      mbar_init(&S.b_empty[i], 1);
    }
    mbar_init(&S.acc_full, 1);
    mbar_init(&S.acc_empty, 8);
    mbar_init(&S.drain, 1);
    S.abort = 0;
    fence_mbar_init();
  }
  if (warp == W_MMA) tmem_alloc(&S.tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_slot;
  volatile int* abort = &S.abort;
  const int n_units = GATEUP ? p.hdr->n_units_gu : p.hdr->n_units_dn;

  if (warp == W_CODE) {
    // ------------------------------------------------------------ code producer
    // (no copy under the MOE_STALL_WEIGHT_COPIES test hook: the consumers' waits run out)
    if (lane == 0 && !(p.status && (p.status->stall & MOE_STALL_WEIGHT_COPIES))) {
      prefetch_tmap(&tm_codes);
      if (p.Is > 0) prefetch_tmap(&tm_scodes);
      uint32_t it = 0;
      uint32_t armed = 0, par = 0;  // per stage: copy issued, its phase parity (bit masks, not local memory)
      bool stop = false;
      for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
        const Unit U = decode_unit<GATEUP>(p, u);
        const CUtensorMap* tm = U.shared ? &tm_scodes : &tm_codes;
        int row0;
        if (GATEUP) row0 = (U.shared ? 0 : U.e * 3 * p.I) + U.f0;
        else row0 = (U.shared ? 0 : U.e * 3 * h) + 2 * h + U.f0;
        const int mstride = U.shared ? p.Is : p.I;  // rows between gate and up
        for (int kc0 = 0; kc0 < U.nkc; kc0 += C::CPS, ++it) {
          const int sc = it % C::SC;
          if (!mbar_wait(&S.code_empty[sc], ((it / C::SC) & 1) ^ 1, abort, WAIT_NS)) {
            note_timeout(p.status, abort, GATEUP ? 11 : 21);
            stop = true;
            break;
          }
          mbar_arrive_expect_tx(&S.code_full[sc], C::C_STAGE);
#pragma unroll
          for (int m = 0; m < C::NMAT; ++m)
            tma_load_2d(c_s + sc * C::C_STAGE + m * 128 * C::CPS * 32, tm, kc0 * 32, row0 + m * mstride,
                        &S.code_full[sc]);
          armed |= 1u << sc;
          par = (par & ~(1u << sc)) | (((it / C::SC) & 1u) << sc);
        }
        if (*abort) stop = true;
      }
      if (*abort)
        for (int i = 0; i < C::SC; ++i)
          if ((armed >> i) & 1u) drain_wait(&S.code_full[i], (par >> i) & 1u);
    }
  } else if (warp == W_B) {
    // ------------------------------------------------------------ B producer
    if (lane == 0) {
      prefetch_tmap(&tm_b);
      if (p.Is > 0) prefetch_tmap(&tm_sb);
    }
    uint32_t it = 0;
    uint32_t armed = 0, par = 0;  // as for the code stages
    for (int u = blockIdx.x; u < n_units && !*abort; u += gridDim.x) {
      const Unit U = decode_unit<GATEUP>(p, u);
      if (GATEUP) {
        __syncwarp();
        for (int i = lane; i < U.Nm; i += 32) {
          const int r = min(i, U.n - 1);
          S.rowidx[i] = U.shared ? U.start + r : p.rows[U.start + r];
        }
        __syncwarp();
      }
      if (lane == 0) {
        const CUtensorMap* tm = U.shared ? &tm_sb : &tm_b;
        for (int kc0 = 0; kc0 < U.nkc; kc0 += U.kps, ++it) {
          const int sb = it % SB;
          if (!mbar_wait(&S.b_empty[sb], ((it / SB) & 1) ^ 1, abort, WAIT_NS)) {
            note_timeout(p.status, abort, GATEUP ? 12 : 22);
            break;
          }
          const int nk = min(U.kps, U.nkc - kc0);
          mbar_arrive_expect_tx(&S.b_full[sb], (uint32_t)(nk * U.Nm * 128));
          uint8_t* bd = b_s + sb * B_STAGE;
          for (int s = 0; s < nk; ++s) {
            uint8_t* sub = bd + s * U.Nm * 128;
            if (GATEUP) {
              for (int g = 0; g < U.Nm / 4; ++g)
                tma_gather4(sub + g * 512, tm, (kc0 + s) * KC, S.rowidx[4 * g], S.rowidx[4 * g + 1],
                            S.rowidx[4 * g + 2], S.rowidx[4 * g + 3], &S.b_full[sb]);
            } else {
              for (int g = 0; g < U.Nm / 16; ++g)
                tma_load_2d(sub + g * 2048, tm, (kc0 + s) * KC, U.start + 16 * g, &S.b_full[sb]);
            }
          }
          armed |= 1u << sb;
          par = (par & ~(1u << sb)) | (((it / SB) & 1u) << sb);
        }
      }
      __syncwarp();
    }
    if (lane == 0 && *abort)
      for (int i = 0; i < SB; ++i)
        if ((armed >> i) & 1u) drain_wait(&S.b_full[i], (par >> i) & 1u);
  } else if (warp == W_MMA) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp walks the loop and waits; one elected lane (the same
    // lane every time, so its commits track its own MMAs) issues.
    {
      uint32_t ait = 0, bit = 0, uit = 0;
      for (int u = blockIdx.x; u < n_units && !__any_sync(0xFFFFFFFFu, *abort); u += gridDim.x, ++uit) {
        const Unit U = decode_unit<GATEUP>(p, u);
        const uint32_t idesc = idesc_bf16(128, U.Nm);
        if (uit > 0 && !__all_sync(0xFFFFFFFFu, mbar_wait(&S.acc_empty, (uit - 1) & 1, abort, WAIT_NS))) {
          if (lane == 0) note_timeout(p.status, abort, GATEUP ? 13 : 23);
          break;
        }
        bool ok = true;
        for (int kc = 0; kc < U.nkc; ++kc) {
          const int sub = kc % U.kps;
          const int sb = bit % SB;
          if (sub == 0 && !__all_sync(0xFFFFFFFFu, mbar_wait(&S.b_full[sb], (bit / SB) & 1, abort, WAIT_NS))) {
            if (lane == 0) note_timeout(p.status, abort, GATEUP ? 14 : 24);
            ok = false;
            break;
          }
          const int sa = ait % SA;
          if (!__all_sync(0xFFFFFFFFu, mbar_wait(&S.a_full[sa], (ait / SA) & 1, abort, WAIT_NS))) {
            if (lane == 0) note_timeout(p.status, abort, GATEUP ? 15 : 25);
            ok = false;
            break;
          }
          const bool last_of_b = sub == U.kps - 1 || kc == U.nkc - 1;
          if (elect_one()) {
            tc_fence_after();
            const uint64_t bd = desc_sw128(smem_u32(b_s + sb * B_STAGE + sub * U.Nm * 128));
#pragma unroll
            for (int m = 0; m < C::NMAT; ++m) {
              const uint64_t ad = desc_sw128(smem_u32(a_s + sa * C::A_STAGE + m * 128 * 128));
#pragma unroll
              for (int kk = 0; kk < KC / 16; ++kk)
                mma_bf16(tmem + m * 256, ad + 2 * kk, bd + 2 * kk, idesc, (kc | kk) != 0);
            }
            mma_commit(&S.a_empty[sa]);
            if (last_of_b) mma_commit(&S.b_empty[sb]);
          }
          __syncwarp();
          ++ait;
          if (last_of_b) ++bit;
        }
        if (!ok) break;
        if (elect_one()) mma_commit(&S.acc_full);
        __syncwarp();
      }
      if (__any_sync(0xFFFFFFFFu, *abort)) {
        if (elect_one()) mma_commit(&S.drain);  // completes once every MMA issued so far has
        __syncwarp();
        drain_wait(&S.drain, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ dequant + epilogue
    const int dw = warp - W_DQ0;         // 0..7
    const int o = (dw & 3) * 32 + lane;  // weight row within the 128-row tile
    const int mtx = GATEUP ? (dw >> 2) : 0;
    const int khalf = GATEUP ? 0 : (dw >> 2);  // down: two threads per row, 32 K each
    const int q = warp & 3;              // this warp's TMEM lane quarter
    const int half = dw >> 2;            // epilogue column half
    uint32_t cit = 0, ait = 0, uit = 0;
    for (int u = blockIdx.x; u < n_units && !*abort; u += gridDim.x, ++uit) {
      const Unit U = decode_unit<GATEUP>(p, u);
      const int K = GATEUP ? h : (U.shared ? p.Is : p.I);
      const int Iu = U.shared ? p.Is : p.I;
      // scale/bias of (row f0 + o, group kc): matrix offset + row offset
      size_t goff;
      if (GATEUP) goff = (size_t)mtx * Iu * (h / KC) + (size_t)(U.f0 + o) * (h / KC);
      else goff = (size_t)2 * Iu * (h / KC) + (size_t)(U.f0 + o) * (K / KC);
      const uint16_t* sp = U.shared ? p.s_scales + goff : p.scales + (size_t)U.e * p.rec_groups + goff;
      const uint16_t* bp = U.shared ? p.s_biases + goff : p.biases + (size_t)U.e * p.rec_groups + goff;
      uint16_t s_cur[4], b_cur[4], s_nxt[4], b_nxt[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        s_cur[j] = j < U.nkc ? __ldg(sp + j) : 0;
        b_cur[j] = j < U.nkc ? __ldg(bp + j) : 0;
      }
      bool ok = true;
      for (int kc0 = 0; kc0 < U.nkc && ok; kc0 += 4) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          s_nxt[j] = kc0 + 4 + j < U.nkc ? __ldg(sp + kc0 + 4 + j) : 0;
          b_nxt[j] = kc0 + 4 + j < U.nkc ? __ldg(bp + kc0 + 4 + j) : 0;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int kc = kc0 + j;
          if (kc >= U.nkc) break;
          const int sub = kc % C::CPS;
          const int sc = cit % C::SC;
          const int sa = ait % SA;
          // warp-uniform verdict (the warp's shared-memory A writes and the
          // arrivals below assume all lanes continue together)
          const bool got = (sub != 0 || mbar_wait(&S.code_full[sc], (cit / C::SC) & 1, abort, WAIT_NS)) &&
                           mbar_wait(&S.a_empty[sa], ((ait / SA) & 1) ^ 1, abort, WAIT_NS);
          if (!__all_sync(0xFFFFFFFFu, got)) {
            if (lane == 0) note_timeout(p.status, abort, GATEUP ? 16 : 26);
            ok = false;
            break;
          }
          const __nv_bfloat162 s2 = bf2_from_half(s_cur[j]);
          const __nv_bfloat162 b2 = bf2_from_half(b_cur[j]);
          const uint8_t* crow = c_s + sc * C::C_STAGE + mtx * 128 * C::CPS * 32 + o * C::CPS * 32 + sub * 32;
          uint8_t* atile = a_s + sa * C::A_STAGE + mtx * 128 * 128;
          if (GATEUP) {
            const uint4 c0 = reinterpret_cast<const uint4*>(crow)[0];
            const uint4 c1 = reinterpret_cast<const uint4*>(crow)[1];
            const uint32_t wd[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            dequant_row_store(wd, s2, b2, atile, o, 0, 8);
          } else {
            const uint4 cw = reinterpret_cast<const uint4*>(crow)[khalf];
            const uint32_t wd[8] = {cw.x, cw.y, cw.z, cw.w, 0u, 0u, 0u, 0u};
            dequant_row_store(wd, s2, b2, atile, o, khalf * 4, 4);
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&S.a_full[sa]);
            if (sub == C::CPS - 1 || kc == U.nkc - 1) mbar_arrive(&S.code_empty[sc]);
          }
          ++ait;
          if (sub == C::CPS - 1 || kc == U.nkc - 1) ++cit;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          s_cur[j] = s_nxt[j];
          b_cur[j] = b_nxt[j];
        }
      }
      if (!ok) break;
      // epilogue.  The per-column row index and routing weight are loaded
      // lane-parallel before the accumulator wait (one load per 32 columns)
      // and broadcast with shuffles, so no global load sits on the
      // TMEM -> store path.
      const int ncw = (U.Nm + 31) / 32;  // 32-column groups
      int col_row[8];
      float col_w[8];
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        col_row[g] = 0;
        col_w[g] = 1.f;
        const int col = g * 32 + lane;
        if (g < ncw && col < U.n) {
          if (GATEUP) {
            col_row[g] = U.start + col;
          } else if (U.shared) {
            col_row[g] = U.start + col;
            col_w[g] = p.gate_vals ? p.gate_vals[U.start + col] : 1.f;
          } else {
            col_row[g] = p.rows[U.start + col];
            col_w[g] = p.weights[U.start + col];
          }
        }
      }
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&S.acc_full, uit & 1, abort, WAIT_NS))) {
        if (lane == 0) note_timeout(p.status, abort, GATEUP ? 17 : 27);
        break;
      }
      tc_fence_after();
      const int feat = U.f0 + q * 32 + lane;
      const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
      if (GATEUP) {
        uint16_t* dst = U.shared ? p.hgs + feat : p.hg + feat;
        for (int c = half; c * 16 < U.Nm; c += 2) {
          uint32_t g[16], v[16];
          tmem_ld16(lane_base + c * 16, g);
          tmem_ld16(lane_base + 256 + c * 16, v);
          tmem_ld_wait();
          tmem_ld_fence(g);
          tmem_ld_fence(v);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = c * 16 + j;
            if (col < U.n)
              dst[(size_t)(U.start + col) * Iu] = f2bf(silu_mul(__uint_as_float(g[j]), __uint_as_float(v[j])));
          }
        }
      } else {
        bool bad_row = false;
        for (int c = half; c * 16 < U.Nm; c += 2) {
          uint32_t y[16];
          tmem_ld16(lane_base + c * 16, y);
          tmem_ld_wait();
          tmem_ld_fence(y);
          const int grp = c >> 1;  // 32-column group holding columns c*16 .. c*16+15
          int rsel = col_row[0];
          float wsel = col_w[0];
#pragma unroll
          for (int g = 1; g < 8; ++g)
            if (g == grp) rsel = col_row[g], wsel = col_w[g];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = c * 16 + j;
            const int src = (c & 1) * 16 + j;  // lane holding this column's row/weight
            const int r = __shfl_sync(0xFFFFFFFFu, rsel, src);
            const float wv = __shfl_sync(0xFFFFFFFFu, wsel, src);
            if (col >= U.n) continue;
            const float yv = __uint_as_float(y[j]);
            if (p.deterministic) {
              if (U.shared) p.acc[(size_t)r * h + feat] = wv * yv;
              else p.ybuf[(size_t)(U.start + col) * h + feat] = yv;
            } else if (r >= 0 && r < p.t) {
              atomicAdd(&p.acc[(size_t)r * h + feat], wv * yv);
            } else {
              bad_row = true;
            }
          }
        }
        if (bad_row && lane == 0) raise_flag(p.status, FLAG_BAD_ROW);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.acc_empty);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == W_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ----------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2D map: width (elements), height (rows), row stride bytes, box {bw, bh}.
cudaError_t make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t width, uint64_t height,
                     uint64_t stride_bytes, uint32_t bw, uint32_t bh, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {width, height};
  cuuint64_t strides[1] = {stride_bytes};
  cuuint32_t box[2] = {bw, bh};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}


}  // namespace

cudaError_t tmap_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t width, uint64_t height,
                    uint64_t stride_bytes, uint32_t bw, uint32_t bh, CUtensorMapSwizzle sw) {
  return make_map(m, base, dt, width, height, stride_bytes, bw, bh, sw);
}

cudaError_t launch_schedule(const TcParams& p, SchedHdr* hdr, int4* tiles, int* units_gu, int max_tiles,
                            int tile_max, cudaStream_t stream) {
  MOE_LAUNCH("schedule", stream,
             launch_k(schedule_kernel, 1, 1024, 0, stream, p, hdr, tiles, units_gu, max_tiles, tile_max));
  return cudaGetLastError();
}

cudaError_t launch_shared_gate(const uint16_t* x, const uint16_t* g, int t, int h, float* out, cudaStream_t stream) {
  MOE_LAUNCH("shared_gate", stream, launch_k(shared_gate_kernel, (t + 7) / 8, 256, 0, stream, x, g, t, h, out));
  return cudaGetLastError();
}

size_t tc_max_tiles(const moe_dims& d) {
  return (size_t)d.t * d.k / TILE_MAX + d.E + d.t / TILE_MAX + 2;
}

size_t tc_sched_bytes(const moe_dims& d) {
  const size_t mt = tc_max_tiles(d);
  const int fmax = (d.inter > d.shared_inter ? d.inter : d.shared_inter) / 128;
  return sizeof(SchedHdr) + mt * sizeof(int4) + mt * fmax * sizeof(int) + (size_t)d.t * sizeof(float) + 256;
}

cudaError_t launch_experts_tc(const ExpertsArgs& a, bool deterministic, cudaStream_t stream) {
  moe_dims d{a.t, a.h, a.I, a.E, a.k, a.Is};
  const size_t mt = tc_max_tiles(d);
  const int fmax = (a.I > a.Is ? a.I : a.Is) / 128;
  SchedHdr* hdr = reinterpret_cast<SchedHdr*>(a.sched);
  int4* tiles = reinterpret_cast<int4*>(a.sched + sizeof(SchedHdr));
  int* units = reinterpret_cast<int*>(tiles + mt);
  float* gate_vals = reinterpret_cast<float*>(units + mt * fmax);

  TcParams p{};
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
  p.scales = a.scales;
  p.biases = a.biases;
  p.rec_groups = a.rec_groups;
  p.s_scales = a.s_scales;
  p.s_biases = a.s_biases;
  p.gate_vals = (a.Is > 0 && a.s_gate) ? gate_vals : nullptr;
  p.acc = a.acc;
  p.hg = a.hg;
  p.hgs = a.hgs;
  p.ybuf = a.ybuf;
  p.hdr = hdr;
  p.tiles = tiles;
  p.units_gu = units;
  p.status = a.status;
  // the fp32 block accumulator starts at zero unless deterministic mode's
  // shared expert writes every element of it
  p.zero_acc = (!deterministic || a.Is == 0) ? 1 : 0;

  CUtensorMap tm_codes_gu, tm_scodes_gu, tm_x, tm_codes_dn, tm_scodes_dn, tm_hg, tm_hgs;
  cudaError_t err;
  const uint64_t h = a.h, I = a.I, Is = a.Is;
  // codes viewed as rows of h/2 bytes (gate/up) or I/2 bytes (down)
  const uint32_t cw_gu = Cfg<true>::CPS * 32, cw_dn = Cfg<false>::CPS * 32;  // code box widths (bytes)
  if ((err = make_map(&tm_codes_gu, a.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, h / 2, (uint64_t)a.E * 3 * I, h / 2,
                      cw_gu, 128, CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
    return err;
  if ((err = make_map(&tm_codes_dn, a.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, I / 2, (uint64_t)a.E * 3 * h, I / 2,
                      cw_dn, 128, CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
    return err;
  if ((err = make_map(&tm_x, a.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h, a.t, h * 2, 64, 1,
                      CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return err;
  if ((err = make_map(&tm_hg, a.hg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, I, (uint64_t)a.t * a.k, I * 2, 64, 16,
                      CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return err;
  if (Is > 0) {
    if ((err = make_map(&tm_scodes_gu, a.s_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, h / 2, 3 * Is, h / 2, cw_gu, 128,
                        CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
      return err;
    if ((err = make_map(&tm_scodes_dn, a.s_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, Is / 2, 3 * h, Is / 2, cw_dn, 128,
                        CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
      return err;
    if ((err = make_map(&tm_hgs, a.hgs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Is, a.t, Is * 2, 64, 16,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
      return err;
  } else {
    tm_scodes_gu = tm_codes_gu;
    tm_scodes_dn = tm_codes_dn;
    tm_hgs = tm_hg;
  }

  if ((err = set_smem_limit_once(expert_gemm_kernel<true>, (int)kernel_smem<true>())) != cudaSuccess) return err;
  if ((err = set_smem_limit_once(expert_gemm_kernel<false>, (int)kernel_smem<false>())) != cudaSuccess) return err;

  if ((err = launch_schedule(p, hdr, tiles, units, (int)mt, TILE_MAX, stream)) != cudaSuccess) return err;
  if (p.gate_vals && (err = launch_shared_gate(a.x, a.s_gate, a.t, a.h, gate_vals, stream)) != cudaSuccess)
    return err;
  const int grid = sm_count();
  MOE_LAUNCH("gateup_tc", stream,
             launch_k(expert_gemm_kernel<true>, grid, KTHREADS, kernel_smem<true>(), stream, tm_codes_gu, tm_scodes_gu,
                                                                                     tm_x, tm_x, p));
  MOE_LAUNCH("down_tc", stream,
             launch_k(expert_gemm_kernel<false>, grid, KTHREADS, kernel_smem<false>(), stream, tm_codes_dn, tm_scodes_dn,
                                                                                       tm_hg, tm_hgs, p));
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  return launch_finalize(a, deterministic, stream);
}

}  // namespace moe

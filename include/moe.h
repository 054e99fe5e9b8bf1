/*
 * moe.h - C ABI of the GB300 (sm_103a) routed mixture-of-experts FFN over a
 * prompt chunk.
 *
 * The operation (cherenkov qwen4_exp engine, rustdoc source pages):
 *   - prefill.rs, pf_layer: the router (router_b) produces, for each of the
 *     t rows, the top-k experts (topk_idx) and their weights (topk_w);
 *   - prefill/experts.rs, prepare_expert_jobs: the (row, slot) pairs are
 *     grouped by expert into a CSR list, expert-ascending and row-ascending;
 *   - prefill/experts.rs, pf_experts: a zeroed block output receives the
 *     shared expert over all rows, then every expert's rows are gathered,
 *     run through the gate and up quantised matmuls, silu(gate)*up and the
 *     down quantised matmul, and scatter-added with their routing weight.
 *   - prefill/experts.rs, Q {w, s, b}: weights are 4-bit affine codes,
 *     W[o][i] = q[o][i] * s[o][i/64] + b[o][i/64].
 *
 * Conventions shared by every entry point
 *   - Every array pointer is a DEVICE pointer on the current CUDA device,
 *     allocated and owned by the caller, unless its description says host;
 *     the library keeps no model state and never allocates, frees or
 *     retains caller memory (the one object it allocates is the streaming
 *     context of moe_streamer_create).
 *   - bf16 and fp16 values are passed as their 16-bit patterns (uint16_t).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls only enqueue work on it: they return before the GPU
 *     has run, never synchronise the host (except moe_read_device_status,
 *     moe_noalloc_read_status and moe_forward_streamed), and results are
 *     valid once the stream has reached that point.
 *   - Return value: MOE_OK (0) or a negative moe_status.  Nothing throws or
 *     aborts across the ABI.  Host-side argument checks run before any work
 *     is enqueued; on failure nothing is enqueued.  moe_last_error() gives a
 *     thread-local message for the last failure on the calling thread.
 *   - Device-side checks (an expert id out of range, a row index out of
 *     range, a bounded wait that gave up) set flags in the workspace and skip
 *     the offending element; moe_read_device_status() reports them.
 *   - Supported shapes: 1 <= t <= 65536; h, inter, shared_inter multiples of
 *     128 (shared_inter may be 0: no shared expert); 1 <= E <= 1024;
 *     1 <= k <= min(E, 16).  Pointers must be 16-byte aligned.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_EINVAL = -1,     /* null or misaligned pointer, unknown flag */
  MOE_ESHAPE = -2,     /* a dimension outside the supported range */
  MOE_EWORKSPACE = -3, /* workspace null or smaller than moe_workspace_bytes() */
  MOE_ECUDA = -4,      /* a CUDA runtime call or kernel launch failed */
  MOE_EDEVICE = -5,    /* a device-side input check failed (bad id or row) */
  MOE_ETIMEOUT = -6    /* a bounded device-side wait gave up */
} moe_status;

/* Problem sizes of one MoE block over one chunk. */
typedef struct {
  int32_t t;            /* rows in the chunk */
  int32_t h;            /* hidden size (input and output width) */
  int32_t inter;        /* routed expert intermediate size */
  int32_t E;            /* number of routed experts */
  int32_t k;            /* experts per row */
  int32_t shared_inter; /* shared expert intermediate size; 0 = none */
  int32_t bits;         /* code width of the expert records: 2, 3, 4 or 8 (0 means 4) */
} moe_dims;

/* The expert-grouped list produced by moe_build_csr (all device, caller-owned). */
typedef struct {
  int32_t* offsets; /* [E+1]: expert e owns list positions offsets[e] .. offsets[e+1]-1 */
  int32_t* rows;    /* [t*k]: row index of each list position */
  float* weights;   /* [t*k]: routing weight of each list position (bit copy of w) */
  int32_t* slot_of; /* [t*k]: list position of pair (r, j), indexed r*k + j */
} moe_csr;

/* Quantised expert weights.  One record per expert, each holding three
 * matrices in this order: gate [inter][h], up [inter][h], down [h][inter].
 * codes:  uint8 [E][3*inter*h*bits/8], each matrix row-major and
 *         K-contiguous; a row's bytes form one little-endian bit string and
 *         code k occupies its bits [k*bits, k*bits + bits) (4 bits: two codes
 *         per byte, the low nibble at the even K index).  bits = dims->bits
 *         (0 means 4); records of 2, 3 or 8 bits go through moe_pack_experts and
 *         the tensor-core kernels (MOE_PACKED_WEIGHTS) only.
 * scales, biases: fp16 [E][3*inter*h/64], per output row and 64-wide K
 *         group, row-major [rows][K/64] per matrix, same matrix order. */
typedef struct {
  const uint8_t* codes;
  const uint16_t* scales;
  const uint16_t* biases;
} moe_qweights;

/* The shared expert: one record of the same layout with inter = shared_inter,
 * plus an optional per-row gate vector (bf16 [h]): when non-NULL, the shared
 * expert's output for row r is scaled by sigmoid(x[r] . gate)
 * (prefill/experts.rs, pf_experts -> shared_add_rows binds the rows and a
 * dense shared-gate tensor). */
typedef struct {
  const uint8_t* codes;
  const uint16_t* scales;
  const uint16_t* biases;
  const uint16_t* gate; /* bf16 [h] or NULL */
} moe_shared;

/* Flags of moe_experts_fwd. */
#define MOE_DETERMINISTIC 0x1u /* fixed-order fp32 reduction per row (bitwise reproducible) */
#define MOE_FORCE_SMALL_T 0x2u /* force the weight-streaming small-t kernels */
#define MOE_FORCE_LARGE_T 0x4u /* force the tensor-core grouped GEMM kernels */
#define MOE_SIMPLE_KERNELS 0x8u /* plain CUDA-core kernels (slow; a cross-check path) */
#define MOE_PACKED_WEIGHTS 0x10u /* experts->codes and shared->codes hold moe_pack_experts output */
#define MOE_FUSED_DECODE 0x20u /* moe_forward: one cooperative launch for decode-shaped chunks */

/* Thread-local message of the last failed call on this thread ("" if none). */
const char* moe_last_error(void);

/* Short name of a status code. */
const char* moe_status_string(int status);

/*
 * Router (prefill.rs, pf_layer -> router_b): logits, top-k and weights.
 *
 *   logit[r][e] = sum_i x[r][i] * wr[e][i]  (+ rbias[e])
 *
 * computed in fp32 from the exact bf16 products in a fixed summation order:
 * lane l of 32 owns the K indices 256*m + 8*l + c (c = 0..7) and sums them
 * from +0, m ascending then c ascending; the 32 lane sums combine as
 * P[l] + P[l xor o] for o = 16, 8, 4, 2, 1.  The bias is added last.
 *   idx[r][0..k-1]: the k largest logits, descending, exact ties to the lower id;
 *   w[r][j] = exp(l_j - l_max) / sum over the row's top-k of exp(l - l_max).
 *
 * x      bf16 [t][h]        wr   bf16 [E][h]      rbias  fp32 [E] or NULL
 * idx    int32 [t][k] out   w    fp32 [t][k] out  logits fp32 [t][E] out or NULL
 *
 * Two implementations, with bit-identical idx and w:
 *   - ws given and logits NULL: tensor-core scores (bf16 MMA, fp32
 *     accumulate) bound every logit to within a proven margin of its
 *     fixed-order value; only the experts that can still reach the top k
 *     are recomputed in the fixed order.  Needs ws of at least
 *     moe_workspace_bytes(dims, 0) bytes (dims.inter and dims.shared_inter
 *     do not change the router's share).  The status block of ws records
 *     the largest observed |score - logit| / margin (float bits at byte
 *     offset 8) and the count of recomputed logits (uint32 at offset 12);
 *     a score outside its margin raises MOE_EDEVICE in
 *     moe_read_device_status (then idx may differ from the fixed order).
 *   - ws NULL or logits requested: one pass that evaluates every logit in
 *     the fixed order (slower; its tile of 8 rows of x, 64 x 256 router
 *     weights and 8 x E logits must fit in 227 KB of shared memory, which
 *     holds for h <= 8192 at E <= 1024; MOE_ESHAPE beyond).
 * Errors: MOE_EINVAL, MOE_ESHAPE, MOE_EWORKSPACE, MOE_ECUDA.
 */
int moe_route_topk(const uint16_t* x, const uint16_t* wr, const float* rbias,
                   const moe_dims* dims, int32_t* idx, float* w, float* logits,
                   void* ws, size_t ws_bytes, void* stream);

/*
 * Grouping (prefill/experts.rs, prepare_expert_jobs): the t*k (row, slot)
 * pairs in expert-ascending, row-ascending order.
 *
 *   offsets[e] = number of pairs routed to experts < e   (offsets[E] = t*k)
 *   rows[p], weights[p]: the row and the bit-copied weight w[r][j] of list
 *       position p; within an expert, rows ascend.
 *   slot_of[r*k + j] = position of pair (r, j).
 *
 * idx int32 [t][k], w fp32 [t][k] in; out fields as in moe_csr.
 * ws: workspace of at least moe_workspace_bytes(dims, 0) bytes (may be shared
 * with moe_experts_fwd on the same stream).  An id outside [0, E) sets the
 * MOE_EDEVICE flag and that pair is dropped.
 * Errors: MOE_EINVAL, MOE_ESHAPE, MOE_EWORKSPACE, MOE_ECUDA.
 */
int moe_build_csr(const int32_t* idx, const float* w, const moe_dims* dims,
                  const moe_csr* csr, void* ws, size_t ws_bytes, void* stream);

/*
 * Router and grouping in one call: exactly the results of moe_route_topk
 * (with ws, logits NULL) followed by moe_build_csr on the same workspace --
 * the same idx, w and csr -- with one launch fewer for t <= 16 rows, where
 * the router's last block also builds the list.  Larger t issue the same
 * launches as the two calls.
 *
 * x, wr, rbias, idx, w as in moe_route_topk; csr as in moe_build_csr; ws of
 * at least moe_workspace_bytes(dims, 0) bytes (required).
 * Errors: MOE_EINVAL, MOE_ESHAPE, MOE_EWORKSPACE, MOE_ECUDA.
 */
int moe_route_csr(const uint16_t* x, const uint16_t* wr, const float* rbias,
                  const moe_dims* dims, int32_t* idx, float* w, const moe_csr* csr,
                  void* ws, size_t ws_bytes, void* stream);

/*
 * Expert FFNs (prefill/experts.rs, pf_experts):
 *
 *   out[r] = g_r * FFN_S(x_r) + sum_j w_rj * FFN_{e_rj}(x_r),
 *   FFN(x) = (silu(x G^T) * (x U^T)) D^T,   silu(z) = z / (1 + exp(-z)),
 *
 * with g_r = sigmoid(x_r . shared->gate) or 1, FFN_S the shared expert (none
 * when dims->shared_inter == 0; `shared` may then be NULL) and the routed
 * terms taken from `csr` (as produced by moe_build_csr).  Weights are
 * dequantised to bf16 (one bf16 fma of the code with the bf16-rounded scale
 * and bias), products accumulate in fp32, silu(gate)*up is rounded to bf16,
 * the block sum accumulates in fp32 and `out` is rounded once to bf16.
 * Without MOE_DETERMINISTIC the routed terms are added with fp32 atomics
 * (summation order varies run to run); with it every row sums its shared
 * term and its k terms in expert-ascending order.  The CUDA path computes
 * silu(z) as z * (1 + tanh(z / 2)) / 2 with the hardware tanh approximation
 * (absolute error of the sigmoid about 2^-12, below the bf16 rounding of the
 * result).
 *
 * Kernel choice (the result meets the same tolerance either way):
 *   - weight-streaming small-t kernels when t <= 16 and t * k * inter / 128
 *     < 64 on packed records (few expert tiles: at inter = 768 and k = 8, a
 *     chunk of one row), < 152 on row-major records, or MOE_FORCE_SMALL_T;
 *   - otherwise the tensor-core grouped kernels (MOE_FORCE_LARGE_T forces
 *     them), on packed weights with MOE_PACKED_WEIGHTS, or on the row-major
 *     records;
 *   - MOE_SIMPLE_KERNELS: plain CUDA-core kernels (a slow cross-check).
 * A call whose workspace status block was never cleared (moe_clear_device_
 * status) may report stale flags; the small-t kernels also keep a completion
 * counter there, so clear a new workspace once before its first use.  After a
 * call that gave up (MOE_ETIMEOUT), the moe_read_device_status that reports
 * it clears the status block, counters included, so the next call starts
 * clean.
 *
 * x bf16 [t][h] in; out bf16 [t][h] out (no residual is added).
 * ws: at least moe_workspace_bytes(dims, flags) bytes.
 * Errors: MOE_EINVAL, MOE_ESHAPE, MOE_EWORKSPACE, MOE_ECUDA.
 */
int moe_experts_fwd(const uint16_t* x, const moe_csr* csr, const moe_qweights* experts,
                    const moe_shared* shared, uint16_t* out, const moe_dims* dims,
                    uint32_t flags, void* ws, size_t ws_bytes, void* stream);

/*
 * The whole block in one call: exactly moe_route_csr followed by
 * moe_experts_fwd on the same workspace and stream -- the same idx, w and
 * csr bit for bit, and `out` within the same tolerance (the fp32 block
 * accumulator is summed in another order).  Arguments as in those two calls.
 *
 * Decode-shaped chunks (decode.rs, step_rows: the MoE block over a verify
 * batch of a few rows) take one launch instead of three with
 * MOE_FUSED_DECODE: when t <= 8, E <= 256, h <= 2048 (x is staged in shared
 * memory), the weights are packed (MOE_PACKED_WEIGHTS) and none of
 * MOE_DETERMINISTIC, MOE_FORCE_SMALL_T, MOE_FORCE_LARGE_T, MOE_SIMPLE_KERNELS
 * is set, a cooperative grid of one CTA per SM computes the router logits,
 * meets at a grid-wide barrier, groups the rows in every CTA, and streams
 * each CTA's share of the touched experts' weight blocks once through the
 * tensor cores (gate/up, then down, with counters in the workspace in place
 * of kernel boundaries).  Without the flag, or for other chunks, the call
 * issues the launches of the two calls.  MOE_FUSED_DECODE is ignored by
 * moe_route_csr and moe_experts_fwd.
 *
 * The grid barrier counts arrivals in the workspace's status block: clear a
 * fresh workspace once (moe_clear_device_status).  Every wait is bounded;
 * after a call that gave up (MOE_ETIMEOUT from moe_read_device_status),
 * that read has cleared the status block and the next call starts clean.
 * Errors: MOE_EINVAL, MOE_ESHAPE, MOE_EWORKSPACE, MOE_ECUDA.
 */
int moe_forward(const uint16_t* x, const uint16_t* wr, const float* rbias, const moe_qweights* experts,
                const moe_shared* shared, const moe_dims* dims, uint32_t flags, int32_t* idx, float* w,
                const moe_csr* csr, uint16_t* out, void* ws, size_t ws_bytes, void* stream);

/*
 * moe_build_csr without a workspace (no counterpart in the method; an
 * interface for callers that cannot allocate device memory, e.g. code running
 * inside someone else's memory pool or under a rule that forbids cudaMalloc on
 * its hot path).  It computes exactly what moe_build_csr computes, into the
 * caller's `csr` arrays, but keeps its scratch in a fixed array inside this
 * library (about 0.8 MB per GPU that loads the library, held until the process
 * exits).  It allocates nothing and calls no allocating routine.
 *
 *   - t*k must not exceed MOE_NOALLOC_MAX_PAIRS (else MOE_ESHAPE, nothing
 *     enqueued); E <= 1024, k <= min(E, 16).
 *   - Every call looks up the array's device address (cudaGetSymbolAddress)
 *     for the current device, so a device reset or a re-created context
 *     leaves no stale address behind.  The first call on a device may load
 *     the library's module: make it before any stream capture.
 *   - All calls share the one array: calls whose GPU work overlaps (other
 *     streams, other threads) race and give wrong results.  Order them on one
 *     stream or synchronise between them.
 *   - An id outside [0, E) drops its pair (slot_of = -1) as in moe_build_csr
 *     and raises a device-side flag in the array's status block, which
 *     moe_noalloc_read_status reports.
 * Errors: MOE_EINVAL, MOE_ESHAPE, MOE_ECUDA.
 */
#define MOE_NOALLOC_MAX_PAIRS 65536
/* Synchronise `stream`, read the status flags of moe_build_csr_noalloc's
 * scratch on the current device and clear them: MOE_OK, MOE_EDEVICE (an id
 * outside [0, E) was dropped since the last read) or MOE_ECUDA.  Reads
 * nothing else; calls on other streams race with it as with the grouping
 * itself. */
int moe_noalloc_read_status(void* stream);

int moe_build_csr_noalloc(const int32_t* idx, const float* w, const moe_dims* dims, const moe_csr* csr,
                          void* stream);

/*
 * Weight packing (a one-time, model-load step; no counterpart in the method).
 * Rewrites row-major 4-bit expert records (the moe_qweights layout) into
 * tile-contiguous blocks that moe_experts_fwd streams with one bulk copy per
 * 64-wide K chunk.  Per record: the gate/up part, for each 128-row feature
 * tile and each 64-wide K chunk, a gate block then an up block; then the
 * down part, for each 128-row tile of h and each 64-wide K chunk of inter, a
 * down block.  A block is 128 rows x 32 bytes of codes (each 32-bit word holds
 * 8 consecutive K: the even ones in its low 16 bits, the odd ones in its high
 * 16 bits, 4 bits each, lowest K first), then 128 bf16 scales, then 128 bf16
 * biases (4608 bytes).  Scales and biases are rounded from fp16 to bf16 (round
 * to nearest even), the rounding the kernels apply anyway.
 *
 * shared = 0: the E routed records (inter); shared = 1: the shared expert's
 * record (shared_inter; scales/biases of moe_shared, passed as moe_qweights).
 * dst: device buffer of at least moe_packed_bytes(dims, shared) bytes,
 * 16-byte aligned.  Pass the packed buffers to moe_experts_fwd in
 * experts->codes / shared->codes with flag MOE_PACKED_WEIGHTS (scales and
 * biases may then be NULL).  Errors: MOE_EINVAL, MOE_ESHAPE, MOE_ECUDA.
 */
size_t moe_packed_bytes(const moe_dims* dims, int shared);
int moe_pack_experts(const moe_qweights* src, const moe_dims* dims, int shared, void* dst, size_t dst_bytes,
                     void* stream);

/*
 * Streamed experts (prefill.rs module doc and its RING / GROUP constants:
 * records stream through a ring of pool slots, a fetch side filling batches
 * ahead of the GPU with two events per batch; prefill/experts.rs,
 * prepare_expert_jobs: the chunk's most-used experts stay resident, the
 * rest take ring slots; pf_experts: the batch protocol).  The routed
 * records (moe_pack_experts output) live in host memory -- on a Grace
 * machine in its LPDDR, read over NVLink-C2C -- and a device buffer of
 * pool_slots + ring_slots record slots holds the resident set and the ring.
 *
 * The residency plan of one chunk (moe_plan_residency; host code only):
 *   1. the experts with rows are ranked by row count, descending, equal
 *      counts in ascending id order; the first pool_slots form the keep set;
 *   2. a kept expert that is not resident takes the lowest free pool slot,
 *      else the slot of the least recently used resident whose expert has
 *      no rows in this chunk (lower slot on ties), which is evicted; with
 *      neither it streams for this chunk.  Residents used by the chunk are
 *      never evicted.  Every pool slot used gets last-use = `call`;
 *   3. in ascending expert order, an expert already resident reads its pool
 *      slot without a copy (batch 0); a newly kept one is copied into its
 *      pool slot; every other expert is copied into ring slot
 *      ring_pos % ring_slots (ring_pos counting the ring jobs);
 *   4. the copies, in that order, form fetch batches 1, 2, ... of `group`
 *      copies each; fetch batch b overwrites ring slots only after batch
 *      wait_for[b] = b - ring_slots / group (when >= 1) has finished.
 * Records read from a pool slot keep the base layout (dims->bits); the
 * ring's transient misses may come from a second store at another code
 * width (prefill/experts.rs, prepare_expert_jobs: "--miss-experts"), which
 * moves fewer bytes over the host link.
 */
typedef struct {
  int32_t pool_slots; /* >= 0: record slots whose contents persist across calls */
  int32_t ring_slots; /* a positive multiple of group: slots refilled by every call */
  int32_t group;      /* >= 1: records per fetch batch */
  int32_t miss_bits;  /* code width of the ring's records: 0 (= dims->bits), 2, 3, 4 or 8 */
} moe_stream_cfg;

/* One chunk's plan; every pointer is a caller-owned HOST array. */
typedef struct {
  int32_t* pool_expert; /* [pool_slots] in/out: expert in each pool slot, -1 = free */
  int64_t* pool_last;   /* [pool_slots] in/out: call number of each slot's last use */
  int32_t* rec;         /* [E] out: record slot of each expert (pool slot, or
                           pool_slots + ring slot); -1 when it has no rows */
  int32_t* batch;       /* [E] out: 0 resident, b >= 1 its fetch batch, -1 no rows */
  int32_t* copy_expert; /* [E] out: experts whose record is copied, in copy order */
  int32_t* copy_slot;   /* [E] out: the record slot each copy writes */
  int32_t* wait_for;    /* [E + 1] out: per batch, the batch it waits for (0 = none) */
  int32_t n_copies;     /* out */
  int32_t n_batches;    /* out: 1 + the number of fetch batches */
} moe_residency_plan;

/* counts: host int32 [E], rows routed to each expert (negative read as 0).
 * `call` must exceed the call numbers already in pool_last.  Host only: no
 * CUDA call, no allocation.  Errors: MOE_EINVAL (null pointer, bad cfg, a
 * pool entry outside [-1, E) or held twice), MOE_ESHAPE (E outside
 * [1, 1024]). */
int moe_plan_residency(const int32_t* counts, int32_t E, const moe_stream_cfg* cfg, int64_t call,
                       moe_residency_plan* plan);

/* Bytes of the device slot buffer for `dims` and `cfg`: pool_slots records
 * at dims->bits, then ring_slots records at the miss width; 0 on bad
 * arguments.  Host only. */
size_t moe_stream_slot_bytes(const moe_dims* dims, const moe_stream_cfg* cfg);

/* A streaming context: the pool table and call counter, a copy stream,
 * the events of the batch protocol, pinned staging for the expert counts
 * and a small device array for the per-chunk record and batch maps.  The
 * one object this library allocates; create it once per model layer and
 * device (it serves the current device at creation).  Errors: MOE_EINVAL,
 * MOE_ESHAPE, MOE_ECUDA. */
typedef struct moe_streamer moe_streamer;
int moe_streamer_create(const moe_dims* dims, const moe_stream_cfg* cfg, moe_streamer** out);
int moe_streamer_destroy(moe_streamer* st); /* synchronises the device first; NULL is a no-op */
/* The pool table: the expert held by each pool slot (-1 = free) into
 * pool_expert[0 .. min(n, pool_slots)); returns that count or a negative
 * moe_status. */
int moe_streamer_pool(const moe_streamer* st, int32_t* pool_expert, int32_t n);

typedef struct {
  int32_t resident; /* experts that read a resident record (no copy) */
  int32_t filled;   /* records copied into pool slots */
  int32_t streamed; /* records copied into ring slots */
  int32_t batches;  /* fetch batches */
  int64_t bytes;    /* bytes copied host -> device (speculative copies included) */
  int32_t prefetched;    /* records fetched speculatively while the chunk was routed */
  int32_t prefetch_used; /* 1 when they were the plan's first fetch batch */
} moe_stream_stats;

/*
 * moe_forward with the routed records streamed from host memory: the same
 * idx, w and csr as moe_route_csr, and `out` within the same tolerance as
 * moe_experts_fwd on the packed records (bit for bit with
 * MOE_DETERMINISTIC: each row sums its terms in the same fixed order).
 * With a miss store, the experts read from ring slots this chunk use its
 * records instead (the chunk's output then depends on the plan).
 *
 *   1. router and grouping on `stream`; the per-expert counts are copied to
 *      the host and the host waits for them (the one point where this call
 *      blocks the host).  Meanwhile the copy stream, once the previous call
 *      has finished on `stream`, fetches again the previous call's first
 *      fetch batch when it held ring records only (the steady state repeats
 *      the plan): if this call's first fetch batch is the same, its copies
 *      are done; if not, the plan's own copies rewrite those slots before
 *      any batch reads them;
 *   2. the residency plan (moe_plan_residency, call numbers 1, 2, ... per
 *      streamer), and the record and batch maps copied to the device;
 *   3. batch 0 (resident experts and the shared expert) runs on `stream`
 *      while the streamer's copy stream fetches batch 1;
 *   4. per fetch batch b: the copy stream waits for event "done" of batch
 *      wait_for[b], issues one host -> device copy per record (one per run
 *      of consecutive experts bound for consecutive slots) and records
 *      event "fetched"; `stream` waits for "fetched", runs the batch's
 *      experts (tile schedule, gather, gate/up, down) and records "done".
 *   5. the last batch finalises `out`.
 * With a miss store of another width, a batch that holds both pool fills
 * and ring records runs as two passes of the expert kernels, one per width.
 *
 * host_records: E packed routed records (moe_packed_bytes(dims, 0) bytes),
 *   in page-locked host memory (cudaHostAlloc) for the copies to run
 *   asynchronously; on a Grace machine any memory the GPU can address.
 *   Pool slots are filled from it.
 * host_miss_records: the miss store, E packed records at the streamer's
 *   miss width, read for every ring slot; NULL (or ignored) when the miss
 *   width equals dims->bits, and ring slots are then filled from
 *   host_records.
 * slots: device buffer of moe_stream_slot_bytes(dims, cfg) bytes, 16-byte
 *   aligned, used only through `st` (its pool slots keep their records
 *   between calls).
 * shared: the packed shared record on the device (MOE_PACKED_WEIGHTS
 *   layout), or NULL when shared_inter == 0.
 * flags: MOE_PACKED_WEIGHTS (required) and optionally MOE_DETERMINISTIC;
 *   the tensor-core kernels always run.  ws: moe_workspace_bytes(dims, flags).
 * stats: host, may be NULL.
 * Calls on one streamer are issued from one thread; each call's work, its
 * copies included, waits for the end of the previous call on the streamer,
 * on whatever stream that call ran.  After a failed call the pool is emptied
 * (the next call refetches).
 * Errors: MOE_EINVAL, MOE_ESHAPE (dims other than the streamer's), MOE_EWORKSPACE,
 * MOE_ECUDA.
 */
int moe_forward_streamed(const uint16_t* x, const uint16_t* wr, const float* rbias, const uint8_t* host_records,
                         const uint8_t* host_miss_records, uint8_t* slots, const moe_shared* shared,
                         const moe_dims* dims, uint32_t flags,
                         int32_t* idx, float* w, const moe_csr* csr, uint16_t* out, void* ws, size_t ws_bytes,
                         moe_streamer* st, void* stream, moe_stream_stats* stats);

/* Workspace bytes needed by moe_build_csr and moe_experts_fwd for `dims` and
 * `flags` (one buffer serves both calls on one stream).  0 on bad dims. */
size_t moe_workspace_bytes(const moe_dims* dims, uint32_t flags);

/* Clear the device-side status flags in `ws` (enqueued on `stream`).
 * Call once on a fresh workspace. */
int moe_clear_device_status(void* ws, void* stream);

/* Synchronise `stream`, read the device-side status flags in `ws` and clear
 * them.  Returns MOE_OK, MOE_EDEVICE (an id or row out of range was seen),
 * MOE_ETIMEOUT or MOE_ECUDA. */
int moe_read_device_status(void* ws, void* stream);

/*
 * Test hook for the bounded device waits (no counterpart in the method).
 * Sets `what` in the status block of `ws` (enqueued on `stream`); until
 * moe_read_device_status clears it, the calls on this workspace make one
 * kind of wait run out instead of completing:
 *   MOE_STALL_WEIGHT_COPIES: the weight producer of the tensor-core expert
 *     kernels (packed and row-major) and of the small-t kernels issues no
 *     copy, so their consumers' waits give up;
 *   MOE_STALL_GRID_BARRIER: the grid barrier of the fused decode launch
 *     waits for one arrival more than the grid has.
 * Each such wait gives up after its limit (2 s of device time), records
 * MOE_ETIMEOUT, and its CTA lets the copies and MMAs in flight land, frees
 * its tensor memory and returns; later calls on a cleared workspace run
 * normally.  Nothing else reads the hook.  Errors: MOE_EWORKSPACE,
 * MOE_EINVAL (unknown bits), MOE_ECUDA.
 */
#define MOE_STALL_WEIGHT_COPIES 0x1u
#define MOE_STALL_GRID_BARRIER 0x2u
int moe_debug_stall(void* ws, uint32_t what, void* stream);

/*
 * Launch accounting (benchmark support; no counterpart in the method).
 * While enabled, every kernel the library launches is counted and
 * bracketed by a pair of CUDA events on the stream it is launched on, so a
 * benchmark can time each kernel inside a longer timed region.  Off by
 * default; enabling adds two event records per launch.
 */
typedef struct {
  char name[48];    /* kernel name */
  int32_t launches; /* launches since the last moe_profile_enable(1) */
  double total_ms;  /* summed event-measured duration of those launches */
} moe_profile_entry;

/* on != 0: clear previous records and start recording; on == 0: stop. */
int moe_profile_enable(int on);

/* Wait for the recorded events and write one entry per distinct kernel
 * (at most max_entries).  Returns the number of entries written (>= 0) or a
 * negative moe_status. */
int moe_profile_read(moe_profile_entry* entries, int max_entries);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */

"""CPU oracle for the routed mixture-of-experts FFN over a prompt chunk.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library (no kernels, headers, tables or helpers); the
only module both sides read is the seeded input generator
``routed_expert_prefill_gb300.synth``, which holds none of the method's
arithmetic.

What it computes, and where the pages define it (cherenkov ``qwen4_exp``
engine, rustdoc source pages):

* ``prefill.rs``, ``pf_layer``: the router (``router_b``) turns the normed
  rows into logits and a top-k list ``topk_idx`` / ``topk_w`` per row.
* ``prefill/experts.rs``, ``prepare_expert_jobs``: rows are bucketed per
  expert, rows outer and slots inner, and the non-empty buckets are
  concatenated in expert order into ``csr_rows`` / ``csr_w``.
* ``prefill/experts.rs``, ``pf_experts``: the block output is zeroed, the
  shared expert (gate ``qmm``, up ``qmm``, ``silu_mul``, down ``qmm``,
  ``shared_add_rows``) runs over every row, then each expert in ascending
  order gathers its rows (``gather_rows``), runs the gate and up quantised
  matmuls, ``silu_mul``, the down quantised matmul, and scatter-adds the
  result times the routing weight (``scatter_add_rows``).
* ``prefill/experts.rs``, ``prepare_expert_jobs``: a job whose record is a
  resident pool record of the base kind keeps the base layout; the ring's
  transient misses take the ``--miss-experts`` store (``experts_fwd``'s
  optional ``miss`` store).
* ``prefill/experts.rs``, ``Q { w, s, b, out, inp }``: affine quantisation,
  ``W[o, i] = q[o, i] * s[o, i // 64] + b[o, i // 64]``, with codes of
  ``l.bits`` bits (``pf_experts`` passes the layout's ``bits`` to every
  quantised matmul; 4 for the base layout, lower for the low-bit stores).

Floating point: everything after the router is fp64 with the exact
dequantised weights and no intermediate rounding; the output is returned in
fp64 (and rounded once to bf16 on request).  The router is fp32 in a fixed
summation order (``route_logits``), because its result decides integers
(the expert ids) that must match the CUDA path bit for bit.

Readings where the pages are silent (the kernels' bodies are not printed):

* logits: dot product in fp32 with the canonical order below, then ``+ bias``.
* top-k: descending logit, exact ties to the lower expert id.
* weights: softmax over the top-k logits (equal to softmax over all E then
  renormalising the top k).
* shared gate (``shared_add_rows`` binds the rows and a dense gate vector):
  a per-row scalar ``sigmoid(x_r . g)``; absent means 1.
* code packing at ``bits`` bits (not printed): each row K-contiguous, least
  significant bit first, code k in bits ``[k*bits, k*bits + bits)`` of the
  row's little-endian bit string; at 4 bits this is two codes per byte with
  the low nibble at the even K index.
"""

from __future__ import annotations

import numpy as np

GROUP = 64
LANES = 32
CHUNK = 8  # contiguous K elements per lane per step in the canonical order


# ---------------------------------------------------------------------------
# Storage conversions (bit patterns in, numbers out)
# ---------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float64 to bf16 bit patterns, round-to-nearest-even, in one step.

    Exact single rounding: the bf16 neighbours of each value are found from
    its float64 bits directly (bf16 has the fp32 exponent range; the inputs
    here are finite and far from overflow and from the subnormal range).
    """
    a = np.asarray(a, np.float64)
    u = a.view(np.uint64)
    sign = (u >> 63).astype(np.uint64)
    mag = u & np.uint64(0x7FFFFFFFFFFFFFFF)
    # float64 has 52 fraction bits, bf16 has 7: drop 45, round to nearest even.
    drop = np.uint64(45)
    half = np.uint64(1) << (drop - np.uint64(1))
    low = mag & ((np.uint64(1) << drop) - np.uint64(1))
    top = mag >> drop
    up = (low > half) | ((low == half) & ((top & np.uint64(1)) == np.uint64(1)))
    top = top + up.astype(np.uint64)
    # Re-bias exponent from float64 (1023) to bf16/fp32 (127): top holds
    # [exp11 | frac7]; zero stays zero.
    exp = (top >> np.uint64(7)).astype(np.int64)
    frac = (top & np.uint64(0x7F)).astype(np.int64)
    e8 = exp - 1023 + 127
    is_zero = exp == 0
    if np.any(~is_zero & ((e8 <= 0) | (e8 >= 255))):
        raise ValueError("value outside the bf16 normal range")
    bits = (sign.astype(np.int64) << 15) | (np.where(is_zero, 0, e8) << 7) | np.where(is_zero, 0, frac)
    return bits.astype(np.uint16)


def unpack_codes(codes: np.ndarray, rows: int, K: int, bits: int = 4) -> np.ndarray:
    """Integer codes q [rows, K] from a row-major record of ``bits``-bit codes:
    each row's bytes read as one little-endian bit string, code k in bits
    [k*bits, k*bits + bits)."""
    c = np.asarray(codes, np.uint8).reshape(rows, K * bits // 8)
    if bits == 4:  # the same bit string read a byte at a time: low nibble first
        q = np.empty((rows, K), np.int64)
        q[:, 0::2] = c & 0x0F
        q[:, 1::2] = c >> 4
        return q
    if bits == 8:
        return c.astype(np.int64)
    bit = np.unpackbits(c, axis=1, bitorder="little").reshape(rows, K, bits).astype(np.int64)
    return (bit << np.arange(bits, dtype=np.int64)).sum(axis=2)


def dequant(codes: np.ndarray, scales: np.ndarray, biases: np.ndarray, rows: int, K: int,
            bits: int = 4) -> np.ndarray:
    """Affine dequantisation of ``bits``-bit codes, exact in float64.

    ``codes``: uint8 [rows, K*bits/8] (see unpack_codes).
    ``scales``/``biases``: float16 [rows, K/64].
    Returns W[o, i] = q[o, i] * s[o, i // 64] + b[o, i // 64]   (experts.rs, ``Q``).
    """
    q = unpack_codes(codes, rows, K, bits).astype(np.float64)
    s = np.asarray(scales, np.float16).reshape(rows, K // GROUP).astype(np.float64)
    b = np.asarray(biases, np.float16).reshape(rows, K // GROUP).astype(np.float64)
    return q * np.repeat(s, GROUP, axis=1) + np.repeat(b, GROUP, axis=1)


def expert_matrices(codes, scales, biases, h: int, inter: int, bits: int = 4):
    """Split one expert record into dequantised gate [I,h], up [I,h], down [h,I]."""
    nb = inter * h * bits // 8
    ng = inter * h // GROUP
    gate = dequant(codes[0:nb], scales[0:ng], biases[0:ng], inter, h, bits)
    up = dequant(codes[nb:2 * nb], scales[ng:2 * ng], biases[ng:2 * ng], inter, h, bits)
    down = dequant(codes[2 * nb:3 * nb], scales[2 * ng:3 * ng], biases[2 * ng:3 * ng], h, inter, bits)
    return gate, up, down


# ---------------------------------------------------------------------------
# Router (prefill.rs, pf_layer -> router_b)
# ---------------------------------------------------------------------------

def route_logits(x_bits: np.ndarray, wr_bits: np.ndarray, rbias: np.ndarray | None = None) -> np.ndarray:
    """Router logits in float32, in the canonical summation order.

    logit[r, e] = sum_i x[r, i] * wr[e, i] (+ rbias[e]);  wr is [E, h].

    bf16 x bf16 products are exact in fp32, so only the order of the fp32
    additions matters.  The canonical order: split K into 32 lanes, lane l
    owning the indices i = 256*m + 8*l + c (c = 0..7); each lane sums its
    products into a float32 starting at +0, m ascending then c ascending;
    the 32 lane sums are then combined pairwise, lane l taking
    P[l] + P[l xor o] for o = 16, 8, 4, 2, 1; lane 0 holds the logit.  The
    bias, when present, is added last in float32.  Indices past h
    contribute nothing (this equals padding with zeros).
    """
    x = bf16_to_f64(x_bits).astype(np.float32)
    wr = bf16_to_f64(wr_bits).astype(np.float32).T  # [h, E]
    t, h = x.shape
    E = wr.shape[1]
    span = LANES * CHUNK
    hp = -(-h // span) * span
    if hp != h:
        x = np.concatenate([x, np.zeros((t, hp - h), np.float32)], axis=1)
        wr = np.concatenate([wr, np.zeros((hp - h, E), np.float32)], axis=0)
    lanes = np.arange(LANES)
    P = np.zeros((t, LANES, E), np.float32)
    for m in range(hp // span):
        for c in range(CHUNK):
            i = span * m + CHUNK * lanes + c            # [32] indices, one per lane
            prod = x[:, i][:, :, None] * wr[i, :][None, :, :]  # exact in fp32
            P = (P + prod).astype(np.float32)
    for o in (16, 8, 4, 2, 1):
        P = (P + P[:, lanes ^ o, :]).astype(np.float32)
    logits = P[:, 0, :]
    if rbias is not None:
        logits = (logits + np.asarray(rbias, np.float32)[None, :]).astype(np.float32)
    return logits


def route_topk(logits: np.ndarray, k: int):
    """Top-k experts per row and their weights.

    idx[r, :] lists the k largest logits in descending order, exact ties to
    the lower expert id.  w[r, j] = exp(l_j - l_max) / sum over the row's
    top-k of exp(l - l_max), computed in float64 and stored as float32.
    """
    logits = np.asarray(logits, np.float32)
    t, E = logits.shape
    idx = np.empty((t, k), np.int32)
    w = np.empty((t, k), np.float32)
    for r in range(t):
        # Sort by (-logit, expert id): a stable sort of -logit keeps lower ids first.
        order = np.argsort(-logits[r].astype(np.float64), kind="stable")[:k]
        idx[r] = order
        l = logits[r, order].astype(np.float64)
        p = np.exp(l - l[0])
        w[r] = (p / p.sum()).astype(np.float32)
    return idx, w


# ---------------------------------------------------------------------------
# Grouping (experts.rs, prepare_expert_jobs)
# ---------------------------------------------------------------------------

def build_csr(idx: np.ndarray, w: np.ndarray, E: int):
    """Group (row, slot) pairs by expert.

    Rows are visited in ascending order and each row's slots in stored order;
    each pair is appended to its expert's list.  The lists are then
    concatenated in ascending expert order.  Returns

    * offsets int32 [E+1]: list of expert e is rows[offsets[e]:offsets[e+1]]
      (empty experts repeat an offset),
    * rows int32 [t*k], weights float32 [t*k] (the routing weight, copied),
    * slot_of int32 [t*k]: position in ``rows`` of the pair (r, j), indexed r*k+j.
    """
    idx = np.asarray(idx)
    t, k = idx.shape
    lists = [[] for _ in range(E)]
    for r in range(t):
        for j in range(k):
            lists[int(idx[r, j])].append((r, j))
    offsets = np.zeros(E + 1, np.int32)
    rows = np.empty(t * k, np.int32)
    weights = np.empty(t * k, np.float32)
    slot_of = np.empty(t * k, np.int32)
    pos = 0
    for e in range(E):
        offsets[e] = pos
        for r, j in lists[e]:
            rows[pos] = r
            weights[pos] = w[r, j]
            slot_of[r * k + j] = pos
            pos += 1
    offsets[E] = pos
    return offsets, rows, weights, slot_of


# ---------------------------------------------------------------------------
# Expert FFNs (experts.rs, pf_experts)
# ---------------------------------------------------------------------------

def silu(z: np.ndarray) -> np.ndarray:
    """z * sigmoid(z) = z / (1 + exp(-z))."""
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def ffn(X: np.ndarray, gate: np.ndarray, up: np.ndarray, down: np.ndarray) -> np.ndarray:
    """(silu(X G^T) * (X U^T)) D^T for rows X [n, h] (fp64)."""
    g = X @ gate.T
    u = X @ up.T
    return (silu(g) * u) @ down.T


def experts_fwd(x_bits, offsets, rows, weights, codes, scales, biases,
                shared_codes, shared_scales, shared_biases, h: int, inter: int,
                shared_inter: int, shared_gate_bits=None, bits: int = 4, miss=None) -> np.ndarray:
    """Block output [t, h] in float64.

    Zeroed output; the shared expert over all rows (times the optional
    per-row gate); then experts in ascending order: gather the expert's rows,
    gate/up, silu*up, down, and add weight * result into the gathered rows.

    ``miss``: optional second record store for the experts that stream
    through the ring (``prefill/experts.rs``, ``prepare_expert_jobs``: a
    job whose record is a resident pool record of the base kind keeps the
    base layout; every other job, the ring's transient misses, takes the
    ``--miss-experts`` layout).  A dict with ``codes``, ``scales``,
    ``biases``, ``bits`` and ``experts``, the ids whose records come from
    this store; the shared expert always uses the base store.
    """
    X = bf16_to_f64(x_bits)
    t = X.shape[0]
    E = len(offsets) - 1
    out = np.zeros((t, h), np.float64)
    sg, su, sd = expert_matrices(shared_codes, shared_scales, shared_biases, h, shared_inter, bits)
    ys = ffn(X, sg, su, sd)
    if shared_gate_bits is not None:
        gvec = bf16_to_f64(shared_gate_bits)
        ys = ys * (1.0 / (1.0 + np.exp(-(X @ gvec))))[:, None]
    out += ys
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a == b:
            continue
        r = np.asarray(rows[a:b], np.int64)
        if miss is not None and e in miss["experts"]:
            G, U, D = expert_matrices(miss["codes"][e], miss["scales"][e], miss["biases"][e], h, inter,
                                      miss["bits"])
        else:
            G, U, D = expert_matrices(codes[e], scales[e], biases[e], h, inter, bits)
        y = ffn(X[r], G, U, D)
        out[r] += np.asarray(weights[a:b], np.float64)[:, None] * y
    return out


def moe_forward(inp: dict, k: int, h: int, inter: int, shared_inter: int, miss=None):
    """Router + grouping + experts over the inputs of ``synth.make_inputs``.

    Returns a dict with logits, idx, w, the CSR arrays, out (fp64) and
    out_bf16 (bit patterns).  ``miss`` as in ``experts_fwd``.
    """
    logits = route_logits(inp["x"], inp["wr"], inp.get("rbias"))
    idx, w = route_topk(logits, k)
    E = inp["wr"].shape[0]
    offsets, rows, weights, slot_of = build_csr(idx, w, E)
    out = experts_fwd(inp["x"], offsets, rows, weights, inp["codes"], inp["scales"],
                      inp["biases"], inp["shared_codes"], inp["shared_scales"],
                      inp["shared_biases"], h, inter, shared_inter, inp.get("shared_gate"),
                      inp.get("bits", 4), miss)
    return dict(logits=logits, idx=idx, w=w, offsets=offsets, rows=rows, weights=weights,
                slot_of=slot_of, out=out, out_bf16=f64_to_bf16(out))

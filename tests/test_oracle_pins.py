"""Pins for the CPU oracle: checks against facts fixed by the pages and by
mathematics, not against the oracle itself.

* hand-derived golden values (tests/golden/*.json) for the router's fp32
  summation order and for the CSR grouping rule of ``prepare_expert_jobs``;
* a closed form: one-hot quantised experts, whose FFN output is a product of
  scalars that pure-Python ``math`` evaluates element by element;
* invariants: top-k weights sum to 1, the CSR is a permutation sorted by
  (expert, row), row-order invariance, zero weights give zero output;
* brute force: per-row direct evaluation with no grouping.
"""

import json
import math
import os

import numpy as np
import pytest

from oracle import moe_oracle as O
from routed_expert_prefill_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(vals):
    return synth.f32_to_bf16_bits(np.asarray(vals, np.float32))


# ---------------------------------------------------------------- storage

def test_bf16_rounding_known_patterns():
    cases = {
        1.0: 0x3F80,
        -2.5: 0xC020,
        1.0 + 2.0 ** -8: 0x3F80,        # tie, even stays
        1.0 + 3 * 2.0 ** -8: 0x3F82,    # tie, rounds up to even
        1.0 + 2.0 ** -8 + 2.0 ** -30: 0x3F81,  # just above the tie (float64 only)
        0.0: 0x0000,
    }
    for v, bits in cases.items():
        assert int(O.f64_to_bf16(np.array([v]))[0]) == bits, v


def test_bf16_rounding_matches_fp32_path_on_fp32_values():
    rng = np.random.default_rng(5)
    a = rng.standard_normal(10000).astype(np.float32)
    np.testing.assert_array_equal(O.f64_to_bf16(a.astype(np.float64)), synth.f32_to_bf16_bits(a))


def test_dequant_nibble_order_and_groups():
    # Row of K = 128: group 0 has s = 0.5, b = -4; group 1 has s = 0.25, b = -1.
    codes = np.full((1, 64), 0x88, np.uint8)
    codes[0, 0] = 0x21      # K0 = 1 (low nibble), K1 = 2 (high nibble)
    codes[0, 32] = 0x8F     # K64 = 15, K65 = 8
    scales = np.array([[0.5, 0.25]], np.float16)
    biases = np.array([[-4.0, -1.0]], np.float16)
    W = O.dequant(codes, scales, biases, 1, 128)
    assert W[0, 0] == -3.5 and W[0, 1] == -3.0
    assert np.all(W[0, 2:64] == 0.0)
    assert W[0, 64] == 2.75 and W[0, 65] == 1.0
    assert np.all(W[0, 66:] == 1.0)


# ---------------------------------------------------------------- router

def test_router_canonical_order_golden():
    g = json.load(open(os.path.join(GOLDEN, "router_order.json")))
    h = g["h"]
    for case in g["cases"]:
        x = np.zeros((1, h), np.float32)
        wr = np.zeros((1, h), np.float32)
        for i, xi, wi in case["terms"]:
            x[0, i] = xi
            wr[0, i] = wi
        got = O.route_logits(_bf16(x), _bf16(wr))
        assert got.dtype == np.float32
        assert float(got[0, 0]) == case["logit"], case["name"]


def test_router_bias_added_after_dot():
    x = np.zeros((1, 256), np.float32)
    wr = np.zeros((2, 256), np.float32)
    x[0, 3] = 2.0
    wr[0, 3] = 0.5
    wr[1, 3] = -1.5
    got = O.route_logits(_bf16(x), _bf16(wr), np.array([0.25, 10.0], np.float32))
    assert got[0, 0] == np.float32(1.25) and got[0, 1] == np.float32(7.0)


def test_router_logits_within_fp32_bound_of_exact():
    rng = np.random.default_rng(1)
    t, h, E = 12, 768, 10  # h not a multiple of 256 exercises the tail
    x = _bf16(rng.standard_normal((t, h)))
    wr = _bf16(rng.standard_normal((E, h)) * 0.02)
    got = O.route_logits(x, wr).astype(np.float64)
    X, W = O.bf16_to_f64(x), O.bf16_to_f64(wr).T
    exact = X @ W
    absum = np.abs(X) @ np.abs(W)
    # <= h/256 + 8 + 5 roundings along any path, each at most 2^-24 relative.
    n = h // 256 * 8 + 8 + 5
    bound = n * 2.0 ** -24 * absum
    assert np.all(np.abs(got - exact) <= bound)
    # and it is not the exact value by accident (order is really fp32)
    assert np.any(got != exact)


def test_topk_ties_and_order_golden():
    logits = np.array([[0.5, 1.0, 1.0, -2.0]], np.float32)
    idx, w = O.route_topk(logits, 2)
    assert idx.tolist() == [[1, 2]]
    assert w.tolist() == [[0.5, 0.5]]
    idx, w = O.route_topk(np.array([[0.0, 1.0, -7.0]], np.float32), 2)
    assert idx.tolist() == [[1, 0]]
    # softmax of (1, 0): sigmoid(1) and sigmoid(-1)
    assert w[0, 0] == np.float32(0.7310585786300049)
    assert w[0, 1] == np.float32(0.2689414213699951)


def test_topk_is_argmax_set_and_weights_normalised():
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((200, 64)).astype(np.float32)
    logits[5, 10] = logits[5, 11] = logits[5].max() + 1  # a tie at the top
    k = 6
    idx, w = O.route_topk(logits, k)
    for r in range(200):
        s = np.sort(logits[r])[::-1]
        assert set(logits[r, idx[r]].tolist()) <= set(s[:k].tolist())
        assert np.all(logits[r, idx[r]] >= s[k - 1])
        assert len(set(idx[r].tolist())) == k
        assert np.all(np.diff(logits[r, idx[r]]) <= 0)
        assert abs(float(w[r].astype(np.float64).sum()) - 1.0) <= 1e-6
        assert np.all(np.diff(w[r]) <= 0)
    assert idx[5, 0] == 10 and idx[5, 1] == 11


# ---------------------------------------------------------------- CSR

def test_csr_golden():
    g = json.load(open(os.path.join(GOLDEN, "csr_tiny.json")))
    idx = np.array(g["idx"], np.int32)
    w = np.array(g["w"], np.float32)
    offsets, rows, weights, slot_of = O.build_csr(idx, w, g["E"])
    assert offsets.tolist() == g["offsets"]
    assert rows.tolist() == g["rows"]
    np.testing.assert_array_equal(weights, np.array(g["weights"], np.float32))
    assert slot_of.tolist() == g["slot_of"]


def test_csr_invariants_random():
    rng = np.random.default_rng(3)
    t, E, k = 300, 40, 5
    idx = np.stack([rng.permutation(E)[:k] for _ in range(t)]).astype(np.int32)
    w = rng.random((t, k)).astype(np.float32)
    offsets, rows, weights, slot_of = O.build_csr(idx, w, E)
    assert offsets[0] == 0 and offsets[E] == t * k and np.all(np.diff(offsets) >= 0)
    assert sorted(slot_of.tolist()) == list(range(t * k))
    for r in range(t):
        for j in range(k):
            p = slot_of[r * k + j]
            e = idx[r, j]
            assert offsets[e] <= p < offsets[e + 1]
            assert rows[p] == r
            assert weights[p].view(np.uint32) == w[r, j].view(np.uint32)
    for e in range(E):
        seg = rows[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)
        assert len(seg) == int((idx == e).sum())


# ---------------------------------------------------------------- experts

def _onehot_record(rng, h, inter):
    """A quantised record whose dequantised gate/up/down are one-hot rows.

    Every code is 8 and every bias is -8*scale, so W = 0, except one code per
    output row, set to q, which gives W[o, pi(o)] = (q - 8) * s[o, pi(o)//64].
    Returns the record and the (pi, value) map of each matrix.
    """
    codes, scales, biases, maps = [], [], [], []
    for rows, K in ((inter, h), (inter, h), (h, inter)):
        q = np.full((rows, K), 8, np.uint8)
        s = rng.uniform(0.25, 2.0, (rows, K // 64)).astype(np.float16)
        b = (s * np.float16(-8)).astype(np.float16)
        pi = rng.integers(0, K, rows)
        qv = rng.choice([0, 1, 3, 6, 9, 12, 15], rows)
        q[np.arange(rows), pi] = qv
        val = (qv.astype(np.float64) - 8.0) * s[np.arange(rows), pi // 64].astype(np.float64)
        codes.append((q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8).ravel())
        scales.append(s.ravel())
        biases.append(b.ravel())
        maps.append((pi, val))
    return np.concatenate(codes), np.concatenate(scales), np.concatenate(biases), maps


def test_ffn_onehot_closed_form():
    rng = np.random.default_rng(4)
    t, h, inter, E, k, Is = 6, 128, 64, 3, 2, 64
    recs = [_onehot_record(rng, h, inter) for _ in range(E)]
    sh = _onehot_record(rng, h, Is)
    x = _bf16(rng.standard_normal((t, h)))
    wr = _bf16(rng.standard_normal((E, h)))
    inp = dict(x=x, wr=wr, rbias=None,
               codes=np.stack([r[0] for r in recs]), scales=np.stack([r[1] for r in recs]),
               biases=np.stack([r[2] for r in recs]),
               shared_codes=sh[0], shared_scales=sh[1], shared_biases=sh[2], shared_gate=None)
    res = O.moe_forward(inp, k, h, inter, Is)
    X = O.bf16_to_f64(x)

    def y(maps, r, f):
        (pg, vg), (pu, vu), (pd, vd) = maps
        o = pd[f]
        g = X[r, pg[o]] * vg[o]
        u = X[r, pu[o]] * vu[o]
        return vd[f] * (g / (1.0 + math.exp(-g))) * u

    for r in range(t):
        for f in range(h):
            want = y(sh[3], r, f)
            for j in range(k):
                want += float(res["w"][r, j]) * y(recs[int(res["idx"][r, j])][3], r, f)
            assert abs(res["out"][r, f] - want) <= 1e-12 * (1 + abs(want)), (r, f)


def test_zero_weights_give_zero_output():
    w = synth.Workload("z", 5, 256, 64, 4, 2, 64, 9)
    inp = synth.make_inputs(w)
    for key in ("codes", "shared_codes"):
        inp[key] = np.full_like(inp[key], 0x88)
    res = O.moe_forward(inp, w.k, w.h, w.inter, w.shared_inter)
    assert np.all(res["out"] == 0.0)


def _per_row_direct(inp, res, w):
    """Brute force: out[r] = FFN_S(x_r) + sum_j w_j FFN_{e_j}(x_r), no grouping."""
    X = O.bf16_to_f64(inp["x"])
    S = O.expert_matrices(inp["shared_codes"], inp["shared_scales"], inp["shared_biases"], w.h, w.shared_inter)
    mats = {}
    out = np.zeros((w.t, w.h))
    for r in range(w.t):
        acc = O.ffn(X[r:r + 1], *S)[0]
        for j in range(w.k):
            e = int(res["idx"][r, j])
            if e not in mats:
                mats[e] = O.expert_matrices(inp["codes"][e], inp["scales"][e], inp["biases"][e], w.h, w.inter)
            acc = acc + float(res["w"][r, j]) * O.ffn(X[r:r + 1], *mats[e])[0]
        out[r] = acc
    return out


def test_brute_force_per_row_matches_grouped():
    w = synth.WORKLOADS["tiny_t16_h256_e8"]
    inp = synth.make_inputs(w)
    res = O.moe_forward(inp, w.k, w.h, w.inter, w.shared_inter)
    direct = _per_row_direct(inp, res, w)
    scale = np.abs(direct).max()
    assert np.abs(res["out"] - direct).max() <= 1e-12 * scale


def test_row_order_invariance():
    w = synth.WORKLOADS["tiny_t16_h256_e8"]
    inp = synth.make_inputs(w)
    res = O.moe_forward(inp, w.k, w.h, w.inter, w.shared_inter)
    perm = np.random.default_rng(7).permutation(w.t)
    inp2 = dict(inp, x=inp["x"][perm])
    res2 = O.moe_forward(inp2, w.k, w.h, w.inter, w.shared_inter)
    np.testing.assert_array_equal(res2["idx"], res["idx"][perm])
    np.testing.assert_array_equal(res2["logits"], res["logits"][perm])
    assert np.abs(res2["out"] - res["out"][perm]).max() <= 1e-12 * np.abs(res["out"]).max()


def test_shared_gate_closed_form():
    # gate vector g = c * e_3: the shared term of row r is scaled by sigmoid(c * x[r, 3]).
    w = synth.Workload("g", 4, 256, 64, 4, 2, 64, 11)
    inp = synth.make_inputs(w)
    gv = np.zeros(256, np.float32)
    gv[3] = 0.75
    res0 = O.moe_forward(inp, w.k, w.h, w.inter, w.shared_inter)
    res1 = O.moe_forward(dict(inp, shared_gate=_bf16(gv)), w.k, w.h, w.inter, w.shared_inter)
    X = O.bf16_to_f64(inp["x"])
    S = O.expert_matrices(inp["shared_codes"], inp["shared_scales"], inp["shared_biases"], w.h, w.shared_inter)
    ys = O.ffn(X, *S)
    for r in range(w.t):
        sig = 1.0 / (1.0 + math.exp(-0.75 * X[r, 3]))
        np.testing.assert_allclose(res1["out"][r], res0["out"][r] - (1.0 - sig) * ys[r], rtol=0, atol=1e-12)


def _record_from_dense(rng, h: int, inter: int):
    """A quantised record built forward from known integer codes: returns the
    record's bytes (this test's own packing: two codes per byte, low nibble at
    the even K index), its fp16 scales and biases (b = -8 s), and the three
    dense matrices W = (q - 8) * s as float64 torch tensors."""
    import torch

    mats, code_bytes, scales, biases = [], [], [], []
    for rows, K in ((inter, h), (inter, h), (h, inter)):
        q = rng.integers(0, 16, size=(rows, K))
        s = rng.uniform(0.005, 0.02, size=(rows, K // 64)).astype(np.float16)
        b = (s * np.float16(-8)).astype(np.float16)
        packed = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
        code_bytes.append(packed.ravel())
        scales.append(s.ravel())
        biases.append(b.ravel())
        s_full = torch.from_numpy(s.astype(np.float64)).repeat_interleave(64, dim=1)
        mats.append((torch.from_numpy(q.astype(np.float64)) - 8.0) * s_full)
    return np.concatenate(code_bytes), np.concatenate(scales), np.concatenate(biases), mats


def test_e1_k1_is_a_dense_ffn_chain():
    """E = 1, k = 1: routing, grouping, gather and weighted scatter reduce to
    the identity, so the block output is the shared FFN plus one dense FFN.
    The expected value is a plain float64 torch matmul chain over matrices
    built from the codes directly (not through the oracle's unpacking)."""
    import torch

    rng = np.random.default_rng(21)
    t, h, inter, Is = 9, 256, 128, 64
    codes, scales, biases, (G, U, D) = _record_from_dense(rng, h, inter)
    s_codes, s_scales, s_biases, (SG, SU, SD) = _record_from_dense(rng, h, Is)
    x = _bf16(rng.standard_normal((t, h)))
    wr = _bf16(rng.standard_normal((1, h)))
    inp = dict(x=x, wr=wr, rbias=None, codes=codes[None], scales=scales[None], biases=biases[None],
               shared_codes=s_codes, shared_scales=s_scales, shared_biases=s_biases, shared_gate=None)
    res = O.moe_forward(inp, 1, h, inter, Is)
    assert np.all(res["idx"] == 0) and np.all(res["w"] == 1.0)
    assert res["offsets"].tolist() == [0, t] and res["rows"].tolist() == list(range(t))
    X = torch.from_numpy(synth.bf16_bits_to_f32(x).astype(np.float64))
    silu = torch.nn.functional.silu
    want = (silu(X @ SG.T) * (X @ SU.T)) @ SD.T + (silu(X @ G.T) * (X @ U.T)) @ D.T
    err = np.abs(res["out"] - want.numpy()).max()
    assert err <= 1e-12 * np.abs(want.numpy()).max()


def test_skewed_recipe_concentrates_rows():
    # Skewed workload routing: a few experts take most slots, many get 0..3 rows.
    w = synth.WORKLOADS["t4096_h2048_e128_skewed"].replace(t=1024)
    inp = synth.make_inputs(w)
    logits = O.route_logits(inp["x"], inp["wr"], inp["rbias"])
    idx, _ = O.route_topk(logits, w.k)
    counts = np.bincount(idx.ravel(), minlength=w.E)
    top8 = np.sort(counts)[::-1][:8].sum()
    assert top8 >= 0.6 * w.t * w.k
    assert (counts <= 3).sum() >= w.E // 2


# ---------------------------------------------------------------------------
# Low-bit layouts (prefill/experts.rs, pf_experts: the quantised matmuls take
# the layout's bits): code k of a row in bits [k*bits, k*bits + bits) of the
# row's little-endian bit string.
# ---------------------------------------------------------------------------

def _pack_bit_by_bit(q: np.ndarray, bits: int) -> np.ndarray:
    """Pack integer codes [rows, K] one bit at a time into bytes, least
    significant bit first (written without numpy's bit routines)."""
    rows, K = q.shape
    out = np.zeros((rows, K * bits // 8), np.uint8)
    for r in range(rows):
        for k in range(K):
            for j in range(bits):
                pos = k * bits + j
                if (int(q[r, k]) >> j) & 1:
                    out[r, pos // 8] |= np.uint8(1 << (pos % 8))
    return out


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_unpack_codes_inverts_a_bit_by_bit_packer(bits):
    rng = np.random.default_rng(bits)
    q = rng.integers(0, 1 << bits, size=(3, 128))
    np.testing.assert_array_equal(O.unpack_codes(_pack_bit_by_bit(q, bits), 3, 128, bits), q)


def test_low_bit_worked_examples():
    # 2 bits: 0xE4 = 0b11100100 holds, from the least significant bit up, 0, 1, 2, 3
    np.testing.assert_array_equal(O.unpack_codes(np.full(16, 0xE4, np.uint8), 1, 64, 2)[0],
                                  np.tile([0, 1, 2, 3], 16))
    # 3 bits: the codes 0..7 occupy bits 0-23; the set bits are 3, 7 | 9, 10,
    # 14, 15 | 17, 19, 20, 21, 22, 23, i.e. the bytes 0x88, 0xC6, 0xFA
    np.testing.assert_array_equal(O.unpack_codes(np.tile(np.array([0x88, 0xC6, 0xFA], np.uint8), 8), 1, 64, 3)[0],
                                  np.tile(np.arange(8), 8))
    # 4 bits: the same string read a byte at a time, low nibble first
    np.testing.assert_array_equal(O.unpack_codes(np.full(32, 0x5A, np.uint8), 1, 64, 4)[0], np.tile([10, 5], 32))


def test_eight_bit_dequant_closed_form():
    rng = np.random.default_rng(8)
    codes = rng.integers(0, 256, size=(2, 128)).astype(np.uint8)
    s = rng.uniform(0.001, 0.002, size=(2, 2)).astype(np.float16)
    b = (s * np.float16(-128)).astype(np.float16)
    w = O.dequant(codes, s, b, 2, 128, 8)
    for r in range(2):
        for i in range(128):
            assert w[r, i] == float(codes[r, i]) * float(s[r, i // 64]) + float(b[r, i // 64])


@pytest.mark.parametrize("bits", [2, 3, 8])
def test_low_bit_record_has_the_width_of_its_codes(bits):
    """A record of a low-bit workload holds 3 * inter * h * bits / 8 bytes of
    codes and dequantises to weights centred like the 4-bit ones."""
    w = synth.Workload("lb", 4, 256, 128, 4, 2, 128, 3, bits=bits)
    inp = synth.make_inputs(w)
    assert inp["codes"].shape == (4, 3 * 128 * 256 * bits // 8) and inp["bits"] == bits
    G, U, D = O.expert_matrices(inp["codes"][0], inp["scales"][0], inp["biases"][0], 256, 128, bits)
    assert G.shape == (128, 256) and U.shape == (128, 256) and D.shape == (256, 128)
    # codes uniform on [0, 2^bits): the mean weight is half a step below
    # zero, within four standard errors of a mean over the G.size weights
    s = inp["scales"][0].astype(np.float64)
    tol = 4 * (2 ** bits / math.sqrt(12)) / math.sqrt(G.size)
    assert abs(G.mean() / s.mean() + 0.5) < tol


# ------------------------------------------------- streamed-miss record store

def _miss_store(w, bits):
    m = synth.make_inputs(w.replace(bits=bits))
    return m["codes"], m["scales"], m["biases"]


def test_miss_store_equal_to_the_base_store_changes_nothing():
    w = synth.WORKLOADS["tiny_t16_h256_e8"]
    inp = synth.make_inputs(w)
    base = O.moe_forward(inp, w.k, w.h, w.inter, w.shared_inter)
    miss = dict(codes=inp["codes"], scales=inp["scales"], biases=inp["biases"], bits=4, experts={0, 3, 5})
    mixed = O.moe_forward(inp, w.k, w.h, w.inter, w.shared_inter, miss=miss)
    np.testing.assert_array_equal(mixed["out"], base["out"])


def test_every_expert_from_a_same_width_miss_store_is_that_store():
    # a second 4-bit store (another draw) serving every routed expert equals
    # the forward pass over that store, with the same shared expert
    w = synth.WORKLOADS["tiny_t16_h256_e8"]
    inp = synth.make_inputs(w)
    other = synth.make_inputs(w.replace(seed=w.seed + 100))
    miss = dict(codes=other["codes"], scales=other["scales"], biases=other["biases"], bits=4,
                experts=set(range(w.E)))
    mixed = O.moe_forward(inp, w.k, w.h, w.inter, w.shared_inter, miss=miss)
    swapped = dict(inp, codes=other["codes"], scales=other["scales"], biases=other["biases"])
    ref = O.moe_forward(swapped, w.k, w.h, w.inter, w.shared_inter)
    np.testing.assert_array_equal(mixed["out"], ref["out"])


def test_mixed_widths_brute_force_per_row():
    # base records at 4 bits, the misses of experts 1, 2 and 6 at 2 bits:
    # each row evaluated directly, with each expert's matrices taken from the
    # store that serves it; and the result differs from both single-store
    # passes (the selection matters)
    w = synth.WORKLOADS["tiny_t16_h256_e8"]
    inp = synth.make_inputs(w)
    mc, ms, mb = _miss_store(w, 2)
    streamed = {1, 2, 6}
    miss = dict(codes=mc, scales=ms, biases=mb, bits=2, experts=streamed)
    res = O.moe_forward(inp, w.k, w.h, w.inter, w.shared_inter, miss=miss)
    X = O.bf16_to_f64(inp["x"])
    S = O.expert_matrices(inp["shared_codes"], inp["shared_scales"], inp["shared_biases"], w.h, w.shared_inter)
    direct = np.zeros((w.t, w.h))
    for r in range(w.t):
        acc = O.ffn(X[r:r + 1], *S)[0]
        for j in range(w.k):
            e = int(res["idx"][r, j])
            if e in streamed:
                m = O.expert_matrices(mc[e], ms[e], mb[e], w.h, w.inter, 2)
            else:
                m = O.expert_matrices(inp["codes"][e], inp["scales"][e], inp["biases"][e], w.h, w.inter)
            acc = acc + float(res["w"][r, j]) * O.ffn(X[r:r + 1], *m)[0]
        direct[r] = acc
    scale = np.abs(direct).max()
    assert np.abs(res["out"] - direct).max() <= 1e-12 * scale
    base = O.moe_forward(inp, w.k, w.h, w.inter, w.shared_inter)
    assert np.abs(res["out"] - base["out"]).max() > 1e-3 * scale
    all_miss = O.moe_forward(inp, w.k, w.h, w.inter, w.shared_inter,
                             miss=dict(miss, experts=set(range(w.E))))
    assert np.abs(res["out"] - all_miss["out"]).max() > 1e-3 * scale

"""The library's residency planner (host code behind moe_plan_residency)
against the oracle's plan, bit for bit, on the worked examples and on random
sequences of chunks; and the argument checks of the streaming entry points
that run before any CUDA call.  No GPU needed."""

import ctypes

import numpy as np
import pytest

from oracle import residency as R

moe = pytest.importorskip("routed_expert_prefill_gb300.moe")


@pytest.fixture(scope="module")
def lib():
    try:
        return moe.load_library()
    except ImportError as e:
        pytest.skip(str(e))


def _same(a, b):
    for key in ("rec", "batch", "copies", "n_batches", "wait_for", "pool_expert", "pool_last"):
        va, vb = a[key], b[key]
        if isinstance(va, int):
            assert va == vb, key
        else:
            assert [tuple(v) if isinstance(v, (list, tuple)) else int(v) for v in va] == \
                [tuple(v) if isinstance(v, (list, tuple)) else int(v) for v in vb], key


@pytest.mark.parametrize("case", [
    ([3, 0, 5, 1, 5, 2], [-1, -1], [0, 0], 1, 4, 2),
    ([4, 6, 0, 0, 1, 0], [2, 4], [1, 1], 2, 4, 2),
    ([2] + [0] * 9, [7, 8, 9], [5, 3, 3], 6, 2, 2),
    ([3, 0, 5, 1, 5, 2], [-1], [0], 1, 2, 1),
    ([0, 2, 0, 7, 1], [], [], 1, 2, 1),
])
def test_worked_examples_match_the_oracle(lib, case):
    counts, pool, last, call, ring, group = case
    _same(moe.plan_residency(counts, pool, last, call, ring, group),
          R.plan(counts, pool, last, call=call, ring=ring, group=group))


@pytest.mark.parametrize("seed", range(30))
def test_random_chunk_sequences_match_the_oracle(lib, seed):
    rng = np.random.default_rng([seed, 902])
    E = int(rng.integers(1, 300))
    P = int(rng.integers(0, E + 4))
    group = int(rng.integers(1, 40))
    ring = group * int(rng.integers(1, 5))
    pool_c = pool_o = [-1] * P
    last_c = last_o = [0] * P
    for call in range(1, 8):
        # a mix of near-uniform and skewed chunks, with unused experts
        if rng.random() < 0.5:
            counts = rng.poisson(4.0, E) * (rng.random(E) < 0.8)
        else:
            counts = (rng.random(E) < 0.5) * rng.zipf(1.5, E).clip(max=4096)
        counts = counts.astype(np.int32)
        c = moe.plan_residency(counts, pool_c, last_c, call, ring, group)
        o = R.plan(counts, pool_o, last_o, call=call, ring=ring, group=group)
        _same(c, o)
        pool_c, last_c = c["pool_expert"], c["pool_last"]
        pool_o, last_o = o["pool_expert"], o["pool_last"]


def test_headline_sized_plan(lib):
    # E = 256 with half the records resident: the first chunk fills the pool
    # with the 128 most-used experts, the next streams only the others
    rng = np.random.default_rng([7, 903])
    counts = rng.multinomial(4096 * 8, np.ones(256) / 256).astype(np.int32)
    p1 = moe.plan_residency(counts, [-1] * 128, [0] * 128, 1, 64, 32)
    _same(p1, R.plan(counts, [-1] * 128, [0] * 128, call=1, ring=64, group=32))
    assert len(p1["copies"]) == 256 and p1["n_batches"] == 9
    p2 = moe.plan_residency(counts, p1["pool_expert"], p1["pool_last"], 2, 64, 32)
    assert len(p2["copies"]) == 128 and p2["n_batches"] == 5
    assert p2["wait_for"] == [0, 0, 0, 1, 2]


def test_plan_argument_checks(lib):
    counts = np.ones(4, np.int32)
    with pytest.raises(moe.MoeError) as e:
        moe.plan_residency(counts, [], [], 1, 3, 2)  # ring not a multiple of the group
    assert e.value.status == -1
    with pytest.raises(moe.MoeError) as e:
        moe.plan_residency(counts, [5], [0], 1, 2, 1)  # pool entry outside [-1, E)
    assert e.value.status == -1
    with pytest.raises(moe.MoeError) as e:
        moe.plan_residency(counts, [1, 1], [0, 0], 1, 2, 1)  # one expert in two slots
    assert e.value.status == -1


def test_streamer_create_rejects_bad_config(lib):
    h = ctypes.c_void_p()
    dims = moe.MoeDims(16, 256, 256, 8, 2, 0, 4)
    for cfg in (moe.MoeStreamCfg(-1, 2, 1), moe.MoeStreamCfg(2, 3, 2), moe.MoeStreamCfg(2, 2, 0)):
        assert lib.moe_streamer_create(ctypes.byref(dims), ctypes.byref(cfg), ctypes.byref(h)) == -1
        assert not h.value
    bad = moe.MoeDims(16, 256, 256, 2000, 2, 0, 4)
    assert lib.moe_streamer_create(ctypes.byref(bad), ctypes.byref(moe.MoeStreamCfg(1, 2, 1)), ctypes.byref(h)) == -2
    assert lib.moe_streamer_destroy(None) == 0


def test_forward_streamed_rejects_a_null_streamer(lib):
    dims = moe.MoeDims(16, 256, 256, 8, 2, 0, 4)
    st = lib.moe_forward_streamed(None, None, None, None, None, None, None, ctypes.byref(dims), moe.MOE_PACKED_WEIGHTS,
                                  None, None, None, None, None, 0, None, None, None)
    assert st == -1


def test_slot_bytes_and_miss_width_checks(lib):
    dims = moe.MoeDims(16, 256, 256, 8, 2, 0, 4)
    rec4 = lib.moe_packed_bytes(ctypes.byref(dims), 0) // 8
    rec2 = lib.moe_packed_bytes(ctypes.byref(moe.MoeDims(16, 256, 256, 8, 2, 0, 2)), 0) // 8
    assert rec2 < rec4
    same = moe.MoeStreamCfg(3, 4, 2, 0)
    assert lib.moe_stream_slot_bytes(ctypes.byref(dims), ctypes.byref(same)) == 7 * rec4
    miss = moe.MoeStreamCfg(3, 4, 2, 2)
    assert lib.moe_stream_slot_bytes(ctypes.byref(dims), ctypes.byref(miss)) == 3 * rec4 + 4 * rec2
    h = ctypes.c_void_p()
    for bad in (1, 5, 16, -2):
        cfg = moe.MoeStreamCfg(3, 4, 2, bad)
        assert lib.moe_stream_slot_bytes(ctypes.byref(dims), ctypes.byref(cfg)) == 0
        assert lib.moe_streamer_create(ctypes.byref(dims), ctypes.byref(cfg), ctypes.byref(h)) == -1
        assert not h.value

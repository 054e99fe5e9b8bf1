"""Streamed experts on the GPU: moe_forward_streamed against the oracle and
against the device-resident path, and its residency bookkeeping against the
oracle's plan (cherenkov ``qwen4_exp``, ``prefill/experts.rs``,
``prepare_expert_jobs`` / ``pf_experts``; ``prefill.rs`` RING / GROUP).

* outputs within the block tolerance of the oracle;
* with MOE_DETERMINISTIC, bit for bit equal to the resident tensor-core
  path: streaming changes where a record is read from, not the arithmetic;
* the pool table and the copy counts after every chunk equal the oracle's
  plan for the chunk's expert counts;
* a ring of one batch (every fetch waits for the batch before it), no pool
  at all, and a pool that holds every expert.
"""

import numpy as np
import pytest

from oracle import moe_oracle as O
from oracle import residency as R
from routed_expert_prefill_gb300 import synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

TOL_REL, TOL_ABS = 1e-2, 1e-3


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from routed_expert_prefill_gb300 import build

    build.build()
    from routed_expert_prefill_gb300 import moe as m

    m.load_library()
    return m


def _dims(moe, w):
    return moe.dims_of(w.t, w.h, w.inter, w.E, w.k, w.shared_inter, w.bits)


def _setup(moe, w, seed_shift=0):
    inp = synth.make_inputs(w.replace(seed=w.seed + seed_shift) if seed_shift else w)
    dev = moe.upload_inputs(inp)
    moe.add_packed(dev, _dims(moe, w))
    return inp, dev


def _streamer(moe, w, dev, pool, ring, group, miss=None):
    host = dev["packed"].cpu().pin_memory()
    if miss is None:
        return moe.Streamer(_dims(moe, w), pool, ring, group, host)
    bits, miss_packed = miss
    return moe.Streamer(_dims(moe, w), pool, ring, group, host, host_miss_records=miss_packed.cpu().pin_memory(),
                        miss_bits=bits)


def _miss_store(moe, w, bits):
    """The miss store: the workload's records drawn at another code width
    (host arrays for the oracle, packed device records for the streamer)."""
    wm = w.replace(bits=bits)
    m = synth.make_inputs(wm)
    dm = moe.upload_inputs(m)
    packed = moe.pack_experts(dm["codes"], dm["scales"], dm["biases"], _dims(moe, wm))
    torch.cuda.synchronize()
    return dict(codes=m["codes"], scales=m["scales"], biases=m["biases"], bits=bits), packed


def _resident(moe, w, dev, flags):
    res = moe.moe_forward(dev, _dims(moe, w), moe.MOE_PACKED_WEIGHTS | moe.MOE_FORCE_LARGE_T | flags)
    torch.cuda.synchronize()
    assert moe.read_device_status(res["ws"]) == 0
    return res


def _streamed(moe, w, dev, st, flags):
    res = moe.moe_forward_streamed(dev, _dims(moe, w), st, moe.MOE_PACKED_WEIGHTS | flags)
    torch.cuda.synchronize()
    assert moe.read_device_status(res["ws"]) == 0
    return res


def _state(pool):
    """The oracle's view of a fresh streamer with `pool` pool slots."""
    return dict(pool=[-1] * pool, last=[0] * pool, spec=[])


def _check_plan(res, st, state, call):
    """Stats and pool table equal the oracle's plan for the chunk's counts;
    the speculative copies are the last call's first fetch batch (when it
    held ring records only) and count as this call's first batch exactly
    when they are its copies.  Returns the state after the call, with the
    experts read from ring slots under "miss"."""
    offs = res["csr"].offsets.cpu().numpy().astype(np.int64)
    counts = np.diff(offs)
    p = R.plan(counts, state["pool"], state["last"], call=call, ring=st.cfg.ring_slots, group=st.cfg.group)
    P = st.cfg.pool_slots
    n_fill = sum(1 for _, s in p["copies"] if s < P)
    first = [(e, sl) for e, sl in p["copies"] if p["batch"][e] == 1]
    s = res["stats"]
    assert s["resident"] == sum(1 for b in p["batch"] if b == 0)
    assert s["filled"] == n_fill
    assert s["streamed"] == len(p["copies"]) - n_fill
    assert s["batches"] == p["n_batches"] - 1
    assert s["prefetched"] == len(state["spec"])
    assert s["prefetch_used"] == int(bool(state["spec"]) and state["spec"] == first)
    wasted = 0 if s["prefetch_used"] else s["prefetched"] * st.miss_rec_bytes
    assert s["bytes"] == n_fill * st.rec_bytes + (len(p["copies"]) - n_fill) * st.miss_rec_bytes + wasted
    assert st.pool() == p["pool_expert"]
    spec = first if first and all(sl >= P for _, sl in first) else []
    return dict(pool=p["pool_expert"], last=p["pool_last"], spec=spec, miss=R.miss_experts(p, P),
                used=s["prefetch_used"])


CASES = [
    # workload, pool slots, ring slots, group
    ("tiny_t16_h256_e8", 2, 4, 2),
    ("t512_h2048_e128", 32, 16, 8),
    ("t4096_h2048_e128_skewed", 16, 32, 16),
]


@pytest.mark.parametrize("name,pool,ring,group", CASES)
def test_streamed_matches_oracle(moe, name, pool, ring, group):
    w = synth.WORKLOADS[name]
    inp, dev = _setup(moe, w)
    st = _streamer(moe, w, dev, pool, ring, group)
    res = _streamed(moe, w, dev, st, 0)
    if w.t <= 512:
        ref = O.moe_forward(inp, w.k, w.h, w.inter, w.shared_inter)
        np.testing.assert_array_equal(res["idx"].cpu().numpy(), ref["idx"])
        rows = np.arange(w.t)
    else:
        rows = np.random.default_rng([w.seed, 77]).choice(w.t, 48, replace=False)
        sub = dict(inp)
        sub["x"] = inp["x"][rows]
        ref = O.moe_forward(sub, w.k, w.h, w.inter, w.shared_inter)
        np.testing.assert_array_equal(res["idx"].cpu().numpy()[rows], ref["idx"])
    got = res["out"].float().cpu().numpy().astype(np.float64)[rows]
    err = np.abs(got - ref["out"]).max()
    tol = TOL_REL * np.abs(ref["out"]).max() + TOL_ABS
    assert err <= tol, f"max|gpu-oracle| = {err:.4g} > {tol:.4g}"
    _check_plan(res, st, _state(pool), 1)
    st.close()


@pytest.mark.parametrize("bits", [2, 3, 8])
@pytest.mark.parametrize("flags", [0, 1])
def test_miss_store_matches_oracle(moe, bits, flags):
    # 4-bit pool records, the ring's misses from a store at `bits`: the first
    # chunk mixes pool fills and ring copies in one batch (two kernel passes,
    # one per width), the second streams only misses; each chunk's output
    # against the oracle with that chunk's misses taken from the miss store
    w = synth.WORKLOADS["t512_h2048_e128"]
    inp, dev = _setup(moe, w)
    miss, miss_packed = _miss_store(moe, w, bits)
    st = _streamer(moe, w, dev, 32, 16, 8, miss=(bits, miss_packed))
    state = _state(32)
    for call in (1, 2):
        res = _streamed(moe, w, dev, st, flags)
        state = _check_plan(res, st, state, call)
        streamed = state["miss"]
        assert 0 < len(streamed) < w.E
        ref = O.moe_forward(inp, w.k, w.h, w.inter, w.shared_inter, miss=dict(miss, experts=streamed))
        got = res["out"].float().cpu().numpy().astype(np.float64)
        err = np.abs(got - ref["out"]).max()
        tol = TOL_REL * np.abs(ref["out"]).max() + TOL_ABS
        assert err <= tol, f"call {call}: max|gpu-oracle| = {err:.4g} > {tol:.4g}"
    st.close()


@pytest.mark.parametrize("name,pool,ring,group", CASES)
def test_streamed_deterministic_equals_resident_bitwise(moe, name, pool, ring, group):
    w = synth.WORKLOADS[name]
    _, dev = _setup(moe, w)
    ref = _resident(moe, w, dev, moe.MOE_DETERMINISTIC)
    st = _streamer(moe, w, dev, pool, ring, group)
    res = _streamed(moe, w, dev, st, moe.MOE_DETERMINISTIC)
    np.testing.assert_array_equal(res["idx"].cpu().numpy(), ref["idx"].cpu().numpy())
    np.testing.assert_array_equal(res["csr"].offsets.cpu().numpy(), ref["csr"].offsets.cpu().numpy())
    np.testing.assert_array_equal(res["out"].view(torch.int16).cpu().numpy(),
                                  ref["out"].view(torch.int16).cpu().numpy())
    st.close()


def test_pool_persists_across_chunks(moe):
    # five chunks of 32 rows (about an eighth of the experts idle in each, so
    # resident records get evicted) through one streamer: every output bit
    # for bit the resident path's, the pool table the oracle's after each
    w = synth.WORKLOADS["t512_h2048_e128"].replace(t=32)
    _, dev = _setup(moe, w)
    x0 = dev["x"]
    st = _streamer(moe, w, dev, 24, 16, 8)
    state = _state(24)
    evicted = 0
    for call in range(1, 6):
        dev["x"] = torch.roll(x0, shifts=call * 5, dims=1).contiguous()  # new rows, new routing
        before = set(state["pool"])
        ref = _resident(moe, w, dev, moe.MOE_DETERMINISTIC)
        res = _streamed(moe, w, dev, st, moe.MOE_DETERMINISTIC)
        np.testing.assert_array_equal(res["out"].view(torch.int16).cpu().numpy(),
                                      ref["out"].view(torch.int16).cpu().numpy())
        state = _check_plan(res, st, state, call)
        evicted += len(before - set(state["pool"]) - {-1})
    assert evicted > 0
    st.close()


@pytest.mark.parametrize("pool,ring,group", [(0, 4, 4), (0, 8, 1), (8, 4, 4)])
def test_single_batch_ring_and_no_pool(moe, pool, ring, group):
    # ring == group: every fetch batch overwrites the slots the previous
    # batch read, so it must wait for that batch; a read before its fetch
    # completed would see another expert's record.  From the second call on
    # the first fetch batch is fetched again while the chunk is routed, into
    # the slots the previous call's last batch read.
    w = synth.WORKLOADS["t512_h2048_e128"]
    _, dev = _setup(moe, w)
    ref = _resident(moe, w, dev, moe.MOE_DETERMINISTIC)
    st = _streamer(moe, w, dev, pool, ring, group)
    state = _state(pool)
    for call in (1, 2, 3):
        res = _streamed(moe, w, dev, st, moe.MOE_DETERMINISTIC)
        np.testing.assert_array_equal(res["out"].view(torch.int16).cpu().numpy(),
                                      ref["out"].view(torch.int16).cpu().numpy())
        state = _check_plan(res, st, state, call)
        if call == 3:
            assert res["stats"]["prefetch_used"] == 1 and res["stats"]["prefetched"] == group
    st.close()


def test_wrong_guess_of_the_first_batch(moe):
    # chunks of 16 rows (a third of the experts idle) whose routing differs
    # from the last one's: the speculative copies of the last call's first
    # batch are then not this call's, and the plan's own copies overwrite
    # those slots before any batch reads them; a repeated chunk uses them
    w = synth.WORKLOADS["t512_h2048_e128"].replace(t=16)
    _, dev = _setup(moe, w)
    x0 = dev["x"]
    st = _streamer(moe, w, dev, 0, 8, 4)
    state = _state(0)
    used = []
    for call, shift in enumerate((0, 7, 7, 13, 29), start=1):
        dev["x"] = torch.roll(x0, shifts=shift, dims=1).contiguous()
        ref = _resident(moe, w, dev, moe.MOE_DETERMINISTIC)
        res = _streamed(moe, w, dev, st, moe.MOE_DETERMINISTIC)
        np.testing.assert_array_equal(res["out"].view(torch.int16).cpu().numpy(),
                                      ref["out"].view(torch.int16).cpu().numpy())
        state = _check_plan(res, st, state, call)
        used.append(state["used"])
    assert used[2] == 1 and 0 in used[1:]
    st.close()


def test_pool_of_every_expert_stops_copying(moe):
    w = synth.WORKLOADS["tiny_t16_h256_e8"]
    _, dev = _setup(moe, w)
    ref = _resident(moe, w, dev, moe.MOE_DETERMINISTIC)
    st = _streamer(moe, w, dev, w.E, 2, 2)
    first = _streamed(moe, w, dev, st, moe.MOE_DETERMINISTIC)
    second = _streamed(moe, w, dev, st, moe.MOE_DETERMINISTIC)
    assert first["stats"]["filled"] == int((first["csr"].offsets.diff() > 0).sum())
    assert second["stats"]["bytes"] == 0 and second["stats"]["batches"] == 0
    for r in (first, second):
        np.testing.assert_array_equal(r["out"].view(torch.int16).cpu().numpy(),
                                      ref["out"].view(torch.int16).cpu().numpy())
    st.close()


@pytest.mark.parametrize("bits", [3, 8])
def test_streamed_low_bit_records(moe, bits):
    w = synth.WORKLOADS["t512_h2048_e128"].replace(bits=bits)
    _, dev = _setup(moe, w)
    ref = _resident(moe, w, dev, moe.MOE_DETERMINISTIC)
    st = _streamer(moe, w, dev, 16, 32, 16)
    res = _streamed(moe, w, dev, st, moe.MOE_DETERMINISTIC)
    np.testing.assert_array_equal(res["out"].view(torch.int16).cpu().numpy(),
                                  ref["out"].view(torch.int16).cpu().numpy())
    st.close()


def test_headline_half_resident(moe):
    # t = 4096, h = 4096, inter = 1536, E = 256, half the records resident
    # after the first chunk.  Deterministic mode bit for bit the resident
    # path's; atomic mode within the tolerance of the oracle on sampled rows.
    w = synth.WORKLOADS["t4096_h4096_e256"]
    inp, dev = _setup(moe, w)
    ref = _resident(moe, w, dev, moe.MOE_DETERMINISTIC)
    st = _streamer(moe, w, dev, 128, 64, 32)
    state = _state(128)
    res = _streamed(moe, w, dev, st, moe.MOE_DETERMINISTIC)
    np.testing.assert_array_equal(res["out"].view(torch.int16).cpu().numpy(),
                                  ref["out"].view(torch.int16).cpu().numpy())
    state = _check_plan(res, st, state, 1)
    res = _streamed(moe, w, dev, st, 0)
    state = _check_plan(res, st, state, 2)
    assert res["stats"]["streamed"] == 128 and res["stats"]["resident"] == 128
    rows = np.random.default_rng([w.seed, 78]).choice(w.t, 16, replace=False)
    sub = dict(inp)
    sub["x"] = inp["x"][rows]
    oref = O.moe_forward(sub, w.k, w.h, w.inter, w.shared_inter)
    got = res["out"].float().cpu().numpy().astype(np.float64)[rows]
    err = np.abs(got - oref["out"]).max()
    tol = TOL_REL * np.abs(oref["out"]).max() + TOL_ABS
    assert err <= tol, f"max|gpu-oracle| = {err:.4g} > {tol:.4g}"
    st.close()


def test_headline_miss_store_two_bits(moe):
    # the headline chunk with 2-bit misses after the first chunk: the oracle
    # on sampled rows with the second chunk's misses from the 2-bit store
    w = synth.WORKLOADS["t4096_h4096_e256"]
    inp, dev = _setup(moe, w)
    miss, miss_packed = _miss_store(moe, w, 2)
    st = _streamer(moe, w, dev, 128, 64, 32, miss=(2, miss_packed))
    state = _state(128)
    for call in (1, 2, 3):
        res = _streamed(moe, w, dev, st, 0)
        state = _check_plan(res, st, state, call)
    streamed = state["miss"]
    # the third chunk repeats the second's plan: its first batch was fetched
    # while it was routed
    assert len(streamed) == 128 and res["stats"]["bytes"] == 128 * st.miss_rec_bytes
    assert res["stats"]["prefetch_used"] == 1
    rows = np.random.default_rng([w.seed, 79]).choice(w.t, 16, replace=False)
    sub = dict(inp)
    sub["x"] = inp["x"][rows]
    oref = O.moe_forward(sub, w.k, w.h, w.inter, w.shared_inter, miss=dict(miss, experts=streamed))
    got = res["out"].float().cpu().numpy().astype(np.float64)[rows]
    err = np.abs(got - oref["out"]).max()
    tol = TOL_REL * np.abs(oref["out"]).max() + TOL_ABS
    assert err <= tol, f"max|gpu-oracle| = {err:.4g} > {tol:.4g}"
    st.close()


def test_calls_on_two_streams_follow_each_other(moe):
    # consecutive calls on one streamer issued on two streams, each with its
    # own workspace and output, the host not waiting between them: every
    # call's work (pool fills, speculative copies, batches) follows the
    # previous call, so every output is the resident path's, bit for bit
    w = synth.WORKLOADS["t512_h2048_e128"].replace(t=32)
    _, dev = _setup(moe, w)
    x0 = dev["x"]
    st = _streamer(moe, w, dev, 24, 8, 4)
    dims = _dims(moe, w)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    xs = [torch.roll(x0, shifts=sh, dims=1).contiguous() for sh in (0, 5, 5, 11, 3, 3)]
    refs = []
    for x in xs:
        dev["x"] = x
        refs.append(_resident(moe, w, dev, moe.MOE_DETERMINISTIC)["out"].clone())
    torch.cuda.synchronize()
    outs = []
    for i, x in enumerate(xs):
        s = streams[i % 2]
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            ws = moe.new_workspace(dims, moe.MOE_PACKED_WEIGHTS | moe.MOE_DETERMINISTIC, stream=s)
            res = moe.moe_forward_streamed(dict(dev, x=x), dims, st,
                                           moe.MOE_PACKED_WEIGHTS | moe.MOE_DETERMINISTIC, ws=ws, stream=s)
            outs.append((res["out"], res["ws"]))
    torch.cuda.synchronize()
    for (o, ws), ref in zip(outs, refs):
        assert moe.read_device_status(ws) == 0
        np.testing.assert_array_equal(o.view(torch.int16).cpu().numpy(), ref.view(torch.int16).cpu().numpy())
    st.close()


@pytest.mark.parametrize("t", [1, 3])
def test_decode_sized_chunks(moe, t):
    # chunks of 1 and 3 rows through the streamed path (the tensor-core
    # kernels on 64-row tiles): bit for bit the resident tensor-core path's,
    # and within the tolerance of the oracle
    w = synth.WORKLOADS["t512_h2048_e128"].replace(t=t)
    inp, dev = _setup(moe, w)
    ref = _resident(moe, w, dev, moe.MOE_DETERMINISTIC)
    st = _streamer(moe, w, dev, 4, 8, 4)
    state = _state(4)
    for call in (1, 2):
        res = _streamed(moe, w, dev, st, moe.MOE_DETERMINISTIC)
        np.testing.assert_array_equal(res["out"].view(torch.int16).cpu().numpy(),
                                      ref["out"].view(torch.int16).cpu().numpy())
        state = _check_plan(res, st, state, call)
    oref = O.moe_forward(inp, w.k, w.h, w.inter, w.shared_inter)
    got = res["out"].float().cpu().numpy().astype(np.float64)
    assert np.abs(got - oref["out"]).max() <= TOL_REL * np.abs(oref["out"]).max() + TOL_ABS
    st.close()


def test_no_shared_expert_and_odd_expert_count(moe):
    # E = 40 (not a multiple of 32), k = 8, no shared expert, t = 300
    w = synth.Workload("st_e40", 300, 512, 256, 40, 8, 0, 91)
    inp, dev = _setup(moe, w)
    ref = _resident(moe, w, dev, moe.MOE_DETERMINISTIC)
    st = _streamer(moe, w, dev, 10, 6, 3)
    state = _state(10)
    for call in (1, 2):
        res = _streamed(moe, w, dev, st, moe.MOE_DETERMINISTIC)
        np.testing.assert_array_equal(res["out"].view(torch.int16).cpu().numpy(),
                                      ref["out"].view(torch.int16).cpu().numpy())
        state = _check_plan(res, st, state, call)
    oref = O.moe_forward(inp, w.k, w.h, w.inter, w.shared_inter)
    got = res["out"].float().cpu().numpy().astype(np.float64)
    assert np.abs(got - oref["out"]).max() <= TOL_REL * np.abs(oref["out"]).max() + TOL_ABS
    st.close()

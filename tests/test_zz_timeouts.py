"""The give-up path of the bounded device waits, exercised on the GPU without
a fault: the test hook moe_debug_stall makes one kind of wait run out (a
producer that issues no copy, a grid barrier that waits for one arrival
more than the grid has).  Each call must come back within its wait limit
(2 s per wait) with MOE_ETIMEOUT from moe_read_device_status, and the same
workspace must then serve a normal call that matches the oracle: the CTAs
that gave up let their copies and MMAs land and freed their tensor memory.

Named to run after the parity tests."""

import time

import numpy as np
import pytest

from oracle import moe_oracle as O
from routed_expert_prefill_gb300 import synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

MOE_ETIMEOUT = -6
LIMIT_S = 20.0  # a few 2 s waits in sequence, plus launch and sync


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from routed_expert_prefill_gb300 import build

    build.build()
    from routed_expert_prefill_gb300 import moe as m

    m.load_library()
    return m


def _check_out(got_bf16, ref_out):
    got = got_bf16.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref_out).max()
    assert err <= 1e-2 * np.abs(ref_out).max() + 1e-3, err


# (workload, flags, stall): the packed tensor-core kernels, the row-major
# tensor-core kernels, the small-t kernels, the fused decode launch
CASES = [
    ("tiny_t16_h256_e8", 0x14, 0x1),  # packed weights, tensor-core kernels forced
    ("tiny_t16_h256_e8", 0x4, 0x1),   # row-major weights, tensor-core kernels forced
    ("decode_t1_h2048_e128", 0x12, 0x1),  # packed weights, small-t kernels forced
    ("decode_t1_h2048_e128", 0x30, 0x2),  # the fused decode launch
]


@pytest.mark.parametrize("name,flags,stall", CASES)
def test_wait_runs_out_and_workspace_recovers(moe, name, flags, stall):
    w = synth.WORKLOADS[name]
    inp = synth.make_inputs(w)
    ref = O.moe_forward(inp, w.k, w.h, w.inter, w.shared_inter)
    dev = moe.upload_inputs(inp)
    dims = moe.dims_of(w.t, w.h, w.inter, w.E, w.k, w.shared_inter)
    if flags & moe.MOE_PACKED_WEIGHTS:
        moe.add_packed(dev, dims)
    ws = moe.new_workspace(dims, flags)

    moe.debug_stall(ws, stall)
    torch.cuda.synchronize()
    t0 = time.monotonic()
    moe.moe_forward(dev, dims, flags, ws=ws)
    status = moe.read_device_status(ws)  # synchronises
    elapsed = time.monotonic() - t0
    assert status == MOE_ETIMEOUT, status
    assert elapsed < LIMIT_S, elapsed

    # the read cleared the hook; the context and the workspace still work
    res = moe.moe_forward(dev, dims, flags, ws=ws)
    assert moe.read_device_status(ws) == 0
    np.testing.assert_array_equal(res["idx"].cpu().numpy(), ref["idx"])
    _check_out(res["out"], ref["out"])


def test_unknown_stall_bits_are_rejected(moe):
    w = synth.WORKLOADS["tiny_t16_h256_e8"]
    dims = moe.dims_of(w.t, w.h, w.inter, w.E, w.k, w.shared_inter)
    ws = moe.new_workspace(dims, 0)
    with pytest.raises(Exception, match="stall"):
        moe.debug_stall(ws, 0x4)
    assert moe.read_device_status(ws) == 0

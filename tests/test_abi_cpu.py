"""The C ABI library loads, exports every symbol include/moe.h declares, and
rejects bad arguments on the host (no GPU needed: these paths return before
any CUDA call)."""

import ctypes
import os
import re

import pytest

from routed_expert_prefill_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    from routed_expert_prefill_gb300 import moe

    return moe.load_library()


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src))


def test_exports_every_declared_symbol(lib):
    from routed_expert_prefill_gb300 import moe

    names = _declared()
    assert names == set(moe.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_bytes(lib):
    from routed_expert_prefill_gb300 import moe

    d = moe.dims_of(512, 2048, 768, 128, 8, 768)
    n0 = lib.moe_workspace_bytes(ctypes.byref(d), 0)
    n1 = lib.moe_workspace_bytes(ctypes.byref(d), moe.MOE_DETERMINISTIC)
    assert n0 >= 512 * 2048 * 4 + 512 * 8 * 768 * 2
    assert n1 >= n0 + 512 * 8 * 2048 * 4
    bad = moe.dims_of(512, 2000, 768, 128, 8, 768)
    assert lib.moe_workspace_bytes(ctypes.byref(bad), 0) == 0


@pytest.mark.parametrize("field,val,status", [
    ("t", 0, -2), ("t", 70000, -2), ("h", 100, -2), ("inter", 96, -2), ("E", 0, -2), ("E", 2000, -2),
    ("k", 0, -2), ("k", 17, -2), ("shared_inter", 64, -2),
])
def test_bad_dims_rejected(lib, field, val, status):
    from routed_expert_prefill_gb300 import moe

    d = moe.dims_of(16, 256, 128, 8, 2, 128)
    setattr(d, field, val)
    fake = ctypes.c_void_p(0x10000)
    rc = lib.moe_route_topk(fake, fake, None, ctypes.byref(d), fake, fake, None, None, 0, None)
    assert rc == status
    assert lib.moe_last_error().decode()


def test_null_and_misaligned_pointers(lib):
    from routed_expert_prefill_gb300 import moe

    d = moe.dims_of(16, 256, 128, 8, 2, 128)
    ok = ctypes.c_void_p(0x10000)
    assert lib.moe_route_topk(None, ok, None, ctypes.byref(d), ok, ok, None, None, 0, None) == -1
    assert lib.moe_route_topk(ctypes.c_void_p(0x10008), ok, None, ctypes.byref(d), ok, ok, None, None, 0, None) == -1
    assert b"aligned" in lib.moe_last_error()
    assert lib.moe_route_topk(ok, ok, None, None, ok, ok, None, None, 0, None) == -1


def test_router_workspace_too_small(lib):
    from routed_expert_prefill_gb300 import moe

    d = moe.dims_of(16, 256, 128, 8, 2, 128)
    ok = ctypes.c_void_p(0x10000)
    need = lib.moe_workspace_bytes(ctypes.byref(d), 0)
    assert lib.moe_route_topk(ok, ok, None, ctypes.byref(d), ok, ok, None, ok, need - 1, None) == -3
    assert b"workspace" in lib.moe_last_error()


def test_workspace_too_small_and_flags(lib):
    from routed_expert_prefill_gb300 import moe

    d = moe.dims_of(16, 256, 128, 8, 2, 128)
    ok = ctypes.c_void_p(0x10000)
    csr = moe.MoeCsr(0x10000, 0x10000, 0x10000, 0x10000)
    assert lib.moe_build_csr(ok, ok, ctypes.byref(d), ctypes.byref(csr), ok, 16, None) == -3
    q = moe.MoeQWeights(0x10000, 0x10000, 0x10000)
    sh = moe.MoeShared(0x10000, 0x10000, 0x10000, None)
    rc = lib.moe_experts_fwd(ok, ctypes.byref(csr), ctypes.byref(q), ctypes.byref(sh), ok, ctypes.byref(d),
                             0x100, ok, 1 << 30, None)
    assert rc == -1 and b"flag" in lib.moe_last_error()
    rc = lib.moe_experts_fwd(ok, ctypes.byref(csr), ctypes.byref(q), None, ok, ctypes.byref(d), 0, ok,
                             1 << 30, None)
    assert rc == -1 and b"shared" in lib.moe_last_error()
    rc = lib.moe_experts_fwd(ok, ctypes.byref(csr), ctypes.byref(q), ctypes.byref(sh), ok, ctypes.byref(d),
                             0, ok, 64, None)
    assert rc == -3


def test_route_csr_argument_checks(lib):
    """moe_route_csr validates like the two calls it combines, before any launch."""
    from routed_expert_prefill_gb300 import moe

    d = moe.dims_of(4, 256, 128, 8, 2, 0)
    ok = ctypes.c_void_p(0x10000)
    csr = moe.MoeCsr(0x10000, 0x10000, 0x10000, 0x10000)
    need = lib.moe_workspace_bytes(ctypes.byref(d), 0)
    assert lib.moe_route_csr(ok, ok, None, ctypes.byref(d), ok, ok, None, ok, need, None) == -1  # csr NULL
    assert lib.moe_route_csr(ok, ok, None, ctypes.byref(d), ok, ok, ctypes.byref(csr), None, 0, None) == -3
    assert lib.moe_route_csr(ok, ok, None, ctypes.byref(d), ok, ok, ctypes.byref(csr), ok, need - 1, None) == -3
    bad = moe.MoeCsr(0x10000, 0x10002, 0x10000, 0x10000)  # misaligned rows
    assert lib.moe_route_csr(ok, ok, None, ctypes.byref(d), ok, ok, ctypes.byref(bad), ok, need, None) == -1
    d.k = 17
    assert lib.moe_route_csr(ok, ok, None, ctypes.byref(d), ok, ok, ctypes.byref(csr), ok, need, None) == -2


def test_status_strings(lib):
    assert lib.moe_status_string(0) == b"MOE_OK"
    assert lib.moe_status_string(-5) == b"MOE_EDEVICE"

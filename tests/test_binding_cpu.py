"""The Python binding rejects, before any call into the library, the argument
errors the C ABI cannot see: the library receives bare pointers, so a wrong
dtype, a strided view, a short output buffer or a tensor on the wrong device
would otherwise become out-of-bounds accesses on the GPU.  CPU only: every
case here raises before a pointer is passed."""

import pytest

torch = pytest.importorskip("torch")

from routed_expert_prefill_gb300 import build as B  # noqa: E402


@pytest.fixture(scope="module")
def moe():
    B.build()
    from routed_expert_prefill_gb300 import moe as m

    m.load_library()
    return m


def _idx_w(t=6, k=2):
    return torch.zeros((t, k), dtype=torch.int32), torch.zeros((t, k), dtype=torch.float32)


def _csr(moe, E, n, short=None):
    sizes = {"offsets": E + 1, "rows": n, "weights": n, "slot_of": n}
    if short:
        sizes[short] -= 1
    return moe.Csr(torch.zeros(sizes["offsets"], dtype=torch.int32), torch.zeros(sizes["rows"], dtype=torch.int32),
                   torch.zeros(sizes["weights"], dtype=torch.float32),
                   torch.zeros(sizes["slot_of"], dtype=torch.int32))


@pytest.mark.parametrize("fn", ["moe_build_csr", "moe_build_csr_noalloc"])
def test_csr_rejects_wrong_dtypes(moe, fn):
    idx, w = _idx_w()
    with pytest.raises(TypeError, match="idx"):
        getattr(moe, fn)(idx.long(), w, 8)
    with pytest.raises(TypeError, match="w must"):
        getattr(moe, fn)(idx, w.double(), 8)


@pytest.mark.parametrize("fn", ["moe_build_csr", "moe_build_csr_noalloc"])
def test_csr_rejects_strided_and_misshaped(moe, fn):
    idx, w = _idx_w()
    strided = torch.zeros((2, 6), dtype=torch.int32).t()  # (6, 2), not contiguous
    with pytest.raises(ValueError, match="contiguous"):
        getattr(moe, fn)(strided, w, 8)
    with pytest.raises(ValueError, match="shape"):
        getattr(moe, fn)(idx, torch.zeros((6, 3), dtype=torch.float32), 8)


@pytest.mark.parametrize("fn", ["moe_build_csr", "moe_build_csr_noalloc"])
@pytest.mark.parametrize("short", ["offsets", "rows", "weights", "slot_of"])
def test_csr_rejects_short_outputs(moe, fn, short):
    idx, w = _idx_w()
    with pytest.raises(ValueError, match=short):
        getattr(moe, fn)(idx, w, 8, out=_csr(moe, 8, 12, short))


@pytest.mark.parametrize("fn", ["moe_build_csr", "moe_build_csr_noalloc"])
def test_csr_rejects_host_tensors(moe, fn):
    idx, w = _idx_w()
    with pytest.raises(ValueError, match="CUDA device"):
        getattr(moe, fn)(idx, w, 8, out=_csr(moe, 8, 12))


def test_router_rejects_bad_inputs(moe):
    x = torch.zeros((4, 256), dtype=torch.bfloat16)
    wr = torch.zeros((8, 256), dtype=torch.bfloat16)
    with pytest.raises(TypeError, match="x must"):
        moe.moe_route_topk(x.float(), wr, 2)
    with pytest.raises(ValueError, match="wr must have shape"):
        moe.moe_route_topk(x, torch.zeros((8, 128), dtype=torch.bfloat16), 2)
    with pytest.raises(ValueError, match="rbias"):
        moe.moe_route_topk(x, wr, 2, rbias=torch.zeros(7))
    with pytest.raises(ValueError, match="idx must have shape"):
        moe.moe_route_topk(x, wr, 2, out=(torch.zeros((4, 3), dtype=torch.int32), torch.zeros((4, 2))))
    with pytest.raises(ValueError, match="CUDA device"):
        moe.moe_route_topk(x, wr, 2, want_logits=True)
    with pytest.raises(ValueError, match="out_csr.rows"):
        moe.moe_route_csr(x, wr, 2, out_csr=_csr(moe, 8, 8, "rows"))


def test_experts_fwd_rejects_bad_inputs(moe):
    dims = moe.dims_of(4, 256, 128, 8, 2, 128)
    x = torch.zeros((4, 256), dtype=torch.bfloat16)
    csr = _csr(moe, 8, 8)
    rec = 3 * 128 * 256
    experts = (torch.zeros(8 * rec // 2, dtype=torch.uint8), torch.zeros(8 * rec // 64, dtype=torch.float16),
               torch.zeros(8 * rec // 64, dtype=torch.float16))
    shared = (torch.zeros(rec // 2, dtype=torch.uint8), torch.zeros(rec // 64, dtype=torch.float16),
              torch.zeros(rec // 64, dtype=torch.float16), None)
    with pytest.raises(ValueError, match="x must have shape"):
        moe.moe_experts_fwd(x[:3], csr, experts, shared, dims, 0)
    with pytest.raises(ValueError, match="experts codes"):
        moe.moe_experts_fwd(x, csr, (experts[0][:-1],) + experts[1:], shared, dims, 0)
    with pytest.raises(TypeError, match="experts scales"):
        moe.moe_experts_fwd(x, csr, (experts[0], experts[1].float(), experts[2]), shared, dims, 0)
    with pytest.raises(ValueError, match="shared expert"):
        moe.moe_experts_fwd(x, csr, experts, None, dims, 0)
    with pytest.raises(ValueError, match="csr.slot_of"):
        moe.moe_experts_fwd(x, _csr(moe, 8, 8, "slot_of"), experts, shared, dims, 0)
    with pytest.raises(ValueError, match="out must have shape"):
        moe.moe_experts_fwd(x, csr, experts, shared, dims, 0, out=torch.zeros((4, 128), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="CUDA device"):
        moe.moe_experts_fwd(x, csr, experts, shared, dims, 0)

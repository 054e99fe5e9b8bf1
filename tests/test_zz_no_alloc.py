"""moe_build_csr_noalloc, the grouping entry point for callers that may not
allocate device memory (it keeps its scratch in a fixed array inside the
library).  Called through the C ABI, it must give exactly what the
workspace-based moe_build_csr gives, on consecutive calls that reuse the same
fixed scratch.  Collected last (file name) so that a run that stops at the
first failure has already run every other test."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from routed_expert_prefill_gb300 import build

    build.build()
    from routed_expert_prefill_gb300 import moe as m

    m.load_library()
    return m


def _routing(t, k, E, seed):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(t)]).astype(np.int32)
    w = rng.random((t, k)).astype(np.float32)
    return torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda()


def _same(got, ref, oracle):
    for name in ("offsets", "rows", "slot_of"):
        np.testing.assert_array_equal(getattr(got, name).cpu().numpy(), getattr(ref, name).cpu().numpy(), name)
    np.testing.assert_array_equal(got.weights.cpu().numpy().view(np.uint32),
                                  ref.weights.cpu().numpy().view(np.uint32))
    # and the grouping the oracle computes from the same ids and weights
    offsets, rows, weights, slot_of = oracle
    np.testing.assert_array_equal(got.offsets.cpu().numpy(), offsets)
    np.testing.assert_array_equal(got.rows.cpu().numpy(), rows)
    np.testing.assert_array_equal(got.slot_of.cpu().numpy(), slot_of)
    np.testing.assert_array_equal(got.weights.cpu().numpy().view(np.uint32), weights.view(np.uint32))


def test_noalloc_csr_matches_workspace_csr_on_consecutive_calls(moe):
    from oracle import moe_oracle as O

    # A large call; a tiny one (one-block path); a smaller one that still
    # takes the multi-block path over the first calls' leftovers; one with a
    # skewed id histogram; and one whose per-chunk count table exactly fills
    # the fixed scratch (E = 1024, 65536 pairs).  Each is checked against the
    # workspace variant and against the oracle's grouping.
    cases = ((4096, 8, 128, 1), (37, 4, 16, 2), (300, 8, 64, 4), (8192, 8, 256, 3), (8192, 8, 1024, 5),
             (300, 8, 64, 6))
    for t, k, E, seed in cases:
        idx, w = _routing(t, k, E, seed)
        if seed == 3:
            idx[: t // 2, 0] = 5  # half the rows share one expert first
            idx[: t // 2, 1:] = torch.where(idx[: t // 2, 1:] == 5, 6, idx[: t // 2, 1:])
        ref = moe.moe_build_csr(idx, w, E)
        got = moe.moe_build_csr_noalloc(idx, w, E)
        torch.cuda.synchronize()
        _same(got, ref, O.build_csr(idx.cpu().numpy(), w.cpu().numpy(), E))


def test_noalloc_rejects_more_pairs_than_its_scratch_holds(moe):
    t, k = 8193, 8  # 65544 pairs > 65536
    idx = torch.zeros((t, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((t, k), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_build_csr_noalloc(idx, w, 16)
    assert ei.value.status == -2
    assert b"scratch" in moe.load_library().moe_last_error()


@pytest.mark.parametrize("t,k,E", [(37, 4, 16), (300, 8, 64)])  # the one-block path and the three-kernel path
def test_noalloc_reports_dropped_ids(moe, t, k, E):
    """An id outside [0, E) drops its pair (slot_of = -1), and the scratch's
    status block reports it to moe_noalloc_read_status until that read clears
    it; a later clean call leaves the status clean."""
    moe.noalloc_read_status()  # clears whatever earlier calls left
    idx, w = _routing(t, k, E, 11)
    idx[3, 1] = E + 7
    got = moe.moe_build_csr_noalloc(idx, w, E)
    ref = moe.moe_build_csr(idx, w, E)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got.slot_of.cpu().numpy(), ref.slot_of.cpu().numpy())
    assert int(got.slot_of.cpu()[3 * k + 1]) == -1
    assert moe.noalloc_read_status() == -5  # MOE_EDEVICE
    assert moe.noalloc_read_status() == 0
    idx2, w2 = _routing(t, k, E, 12)
    moe.moe_build_csr_noalloc(idx2, w2, E)
    assert moe.noalloc_read_status() == 0

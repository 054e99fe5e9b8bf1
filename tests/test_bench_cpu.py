"""The benchmark's output contract and its host-side arithmetic, on CPU.

The reference arm times the oracle alone, so it runs without a GPU; its JSON
line must carry the keys the benchmark contract names.  The GPU arm's helpers
(work model, whole-job throughput, max over ranks) are plain host code.
"""

import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from routed_expert_prefill_gb300 import synth  # noqa: E402


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny_t16_h256_e8", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"] == "tiny_t16_h256_e8"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
    # ms_per_step is the measured time of one step, the oracle over the rows it ran
    rows = d["config"]["rows_per_step"]
    assert 1 <= rows <= d["config"]["t"]
    assert d["ms_per_step"] == pytest.approx(1e3 * rows / d["value"], rel=1e-6)
    assert cb["cores"] == bench.host_cores()


def test_step_work_counts():
    """Flops and bytes of the work model on a hand-checked tiny case."""
    w = synth.Workload("m", 4, 256, 128, 4, 2, 128, 1)
    counts = np.array([3, 0, 4, 1])  # 8 pairs, 3 experts touched
    work = bench.step_work(w, counts)
    n, t, h, inter, si = 8, 4, 256, 128, 128
    gu = 4 * n * h * inter + 4 * t * h * si
    dn = 2 * n * h * inter + 2 * t * h * si
    router = 2 * t * h * w.E
    assert work["touched"] == 3 and work["pairs"] == 8 and work["max_rows"] == 4
    assert work["by_kernel"]["gateup"]["flops"] == gu
    assert work["by_kernel"]["down"]["flops"] == dn
    assert work["flops"] == gu + dn + router
    rec = 3 * h * inter * (1 / 2 + 4 / 64)
    assert work["bytes"] >= 4 * rec  # three touched records and the shared one, plus activations


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_step_work_bytes_follow_the_code_width(bits):
    """Weight bytes of the work model at each code width: bits/8 bytes per
    weight plus a 2-byte scale and bias per 64 weights, for the touched
    records and the shared one; flops do not depend on the width."""
    w = synth.Workload("m", 4, 256, 128, 4, 2, 128, 1, bits=bits)
    w4 = synth.Workload("m", 4, 256, 128, 4, 2, 128, 1)
    counts = np.array([3, 0, 4, 1])
    work, work4 = bench.step_work(w, counts), bench.step_work(w4, counts)
    h, inter = 256, 128
    per_weight = bits / 8 + 4 / 64
    assert bench.record_bytes(h, inter, bits) == 3 * h * inter * per_weight
    assert work["by_kernel"]["gateup"]["bytes"] - work4["by_kernel"]["gateup"]["bytes"] == (
        (3 + 1) * 2 * h * inter * (bits - 4) // 8)
    assert work["by_kernel"]["down"]["bytes"] - work4["by_kernel"]["down"]["bytes"] == (
        (3 + 1) * h * inter * (bits - 4) // 8)
    assert work["flops"] == work4["flops"]


def test_low_bit_headline_workloads_exist():
    for b in (2, 3, 8):
        w = synth.WORKLOADS[f"t4096_h4096_e256_b{b}"]
        base = synth.WORKLOADS["t4096_h4096_e256"]
        assert w.bits == b and (w.t, w.h, w.inter, w.E, w.k, w.shared_inter, w.seed) == (
            base.t, base.h, base.inter, base.E, base.k, base.shared_inter, base.seed)


def test_job_throughput_and_single_rank_max():
    # every rank processes its own chunk: value = world * rows / max time
    assert bench.job_tokens_per_s(1, 512, 0.2) == pytest.approx(512 / 0.2e-3)
    assert bench.job_tokens_per_s(4, 512, 0.2) == pytest.approx(4 * 512 / 0.2e-3)
    assert bench.max_over_ranks(3.5, "cpu") == 3.5


def test_measured_traffic_is_tied_to_the_kernel_sources():
    assert bench.measured_traffic("no_such_workload", "gateup", 16) is None
    for (wl, fam, fl), m in bench.MEASURED_TRAFFIC.items():
        got = bench.measured_traffic(wl, fam, fl)
        assert got is None or got == m["bytes"]


def test_oracle_pool_rows_and_time():
    """The pooled oracle runs the whole sample, split over the cores, in one timed pass."""
    w = synth.WORKLOADS["tiny_t16_h256_e8"]
    pool = bench.OraclePool(w, synth.make_inputs(w), 2)
    try:
        assert pool.seconds(5) > 0
        assert 4 <= pool.rows_for(0.01) <= w.t
    finally:
        pool.close()


def test_step_roofline_picks_the_slower_bound():
    peaks = {"bf16_tflops": 2000.0, "hbm_gbs": 8000.0}
    sr = bench.step_roofline({"flops": 2e12, "bytes": 8e9}, 2.0, peaks)  # 1.0 ms tensor, 1.0 ms HBM
    assert sr["frac"] == pytest.approx(0.5)
    sr = bench.step_roofline({"flops": 4e12, "bytes": 8e9}, 4.0, peaks)
    assert sr["bound"] == "tensor" and sr["frac"] == pytest.approx(0.5)


def test_streamed_entries_follow_the_pages_ring():
    # the streamed bench entries stream the headline chunk through the pages'
    # ring (prefill.rs: RING = 64 slots, GROUP = 8 experts per batch) with
    # half of the 256 records resident, and the miss entry uses 2-bit records
    assert bench.STREAMED_CFG == dict(pool_slots=128, ring_slots=64, group=8)
    assert bench.STREAMED != bench.STREAMED_MISS2
    assert bench.DEFAULT_WORKLOAD == "t4096_h4096_e256"
    assert synth.WORKLOADS[bench.DEFAULT_WORKLOAD].E == 2 * bench.STREAMED_CFG["pool_slots"]
    assert "t4096_h4096_e256_b2" in synth.WORKLOADS

"""Benchmark of the routed-MoE FFN over one prompt chunk on GB300.

A step is one pass of the whole path over one chunk: router top-k, CSR
grouping, and the expert FFNs (shared expert, gate/up + silu*up, down +
weighted scatter-add), i.e. moe_route_topk -> moe_build_csr ->
moe_experts_fwd on one stream.  Inputs are synthetic (routed_expert_prefill_gb300.synth)
and resident in HBM for ``value``; ``e2e`` copies x in from pinned host
memory and the block output back every step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Multi-GPU (torchrun): every rank runs its own chunk (weak scaling, no
collective on the data path); value = chunks' rows over the max-over-ranks time.
"""

import os

# The CPU oracle legs run single-threaded (their reported core count is 1).
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import hashlib
import json
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from routed_expert_prefill_gb300 import synth  # noqa: E402

METRIC = "prefill tokens/s and % of roofline (tensor or HBM) for routed MoE FFN, 1 GB300"
DEFAULT_WORKLOAD = "t512_h2048_e128"
L2_BYTES = 129 * 2 ** 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------------------
# Algorithmic work of one step (from the step's actual routing)
# --------------------------------------------------------------------------

def record_bytes(h, inter):
    """Bytes of one quantised expert record: 4-bit codes + fp16 scale and bias per 64."""
    return 3 * inter * h // 2 + 2 * 2 * (3 * inter * h // 64)


def step_work(w: synth.Workload, counts: np.ndarray) -> dict:
    touched = int((counts > 0).sum())
    n = int(counts.sum())
    t, h, I, Is, E, k = w.t, w.h, w.inter, w.shared_inter, w.E, w.k
    flops = 2 * t * h * E + 6 * n * h * I + 6 * t * h * Is
    wbytes = touched * record_bytes(h, I) + (record_bytes(h, Is) if Is else 0)
    io = 2 * t * h * 2 + E * h * 2 + t * k * 8
    by_kernel = {
        # gate+up weights of touched experts (and the shared expert) + x in + hg out
        "gateup": dict(bytes=touched * 2 * (I * h // 2 + 2 * 2 * I * h // 64)
                       + (2 * (Is * h // 2 + 2 * 2 * Is * h // 64) if Is else 0)
                       + t * h * 2 + (n * I + t * Is) * 2,
                       flops=4 * n * h * I + 4 * t * h * Is),
        # down weights + hg in + fp32 block accumulator in/out
        "down": dict(bytes=touched * (I * h // 2 + 2 * 2 * I * h // 64)
                     + ((Is * h // 2 + 2 * 2 * Is * h // 64) if Is else 0)
                     + (n * I + t * Is) * 2 + 2 * t * h * 4,
                     flops=2 * n * h * I + 2 * t * h * Is),
        # router (scores + exact refinement): x and router weights in, idx/w out
        "route": dict(bytes=t * h * 2 + E * h * 2 + t * k * 8, flops=2 * t * h * E),
    }
    return dict(touched=touched, pairs=n, max_rows=int(counts.max()), flops=flops,
                bytes=wbytes + io, by_kernel=by_kernel)


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of
# the packed expert kernels, from one ncu capture of
# `python bench.py --steps 5 --warmup 3 --no-cpu-baseline [--workload ...]`
# on a GB300; valid
# while the kernel sources hash to `src` (reported as null otherwise).
PACKED_SOURCES = ("experts_packed.cu", "tc_ptx.cuh", "tc_common.cuh", "common.cuh", "experts.cuh")
MEASURED_TRAFFIC = {
    ("t512_h2048_e128", "gateup", 16): dict(bytes=264.25e6, src="59dce5c721bcb98c"),
    ("t512_h2048_e128", "down", 16): dict(bytes=130.16e6, src="59dce5c721bcb98c"),
    ("t4096_h2048_e128_skewed", "gateup", 16): dict(bytes=301.81e6, src="59dce5c721bcb98c"),
    ("t4096_h2048_e128_skewed", "down", 16): dict(bytes=139.19e6, src="59dce5c721bcb98c"),
}


def packed_source_hash() -> str:
    h = hashlib.sha256()
    for f in PACKED_SOURCES:
        with open(os.path.join(ROOT, "routed_expert_prefill_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str, family: str, flags: int):
    m = MEASURED_TRAFFIC.get((workload, family, flags))
    if m is None or m["src"] != packed_source_hash():
        return None
    return m["bytes"]


def max_over_ranks(x: float, device) -> float:
    """The largest x over all ranks of the process group (x itself when alone)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    tt = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_tokens_per_s(world: int, rows_per_rank: int, max_ms: float) -> float:
    """Whole-job throughput: every rank processes its own chunk of rows_per_rank rows."""
    return world * rows_per_rank / (max_ms * 1e-3)


def kernel_family(name: str) -> str:
    for fam in ("gateup", "down", "route"):
        if name.startswith(fam):
            return fam
    return name


# --------------------------------------------------------------------------
# Clocks during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        for ln in self.lines:
            f = [s.strip() for s in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                                 f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------
# Reference arm: the CPU oracle as it stands
# --------------------------------------------------------------------------

def oracle_sample_seconds(w: synth.Workload, inp: dict, rows: int) -> float:
    from oracle import moe_oracle as O

    sub = dict(inp, x=inp["x"][:rows])
    t0 = time.perf_counter()
    O.moe_forward(sub, w.k, w.h, w.inter, w.shared_inter)
    return time.perf_counter() - t0


def calibrated_rows(w: synth.Workload, inp: dict, budget_s: float) -> int:
    """Rows of the workload whose oracle pass takes about budget_s (from a timed 4-row probe)."""
    probe = min(w.t, 4)
    per_row = oracle_sample_seconds(w, inp, probe) / probe
    return int(max(probe, min(w.t, budget_s / max(per_row, 1e-9))))


def run_reference(args, w: synth.Workload):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    inp = synth.make_inputs(w)
    # each step a bounded sample: the whole run stays within about 150 s
    per_step = min(10.0, 150.0 / max(1, args.steps + args.warmup))
    rows = min(calibrated_rows(w, inp, per_step), args.oracle_rows) if args.oracle_rows else \
        calibrated_rows(w, inp, per_step)
    for _ in range(args.warmup):
        oracle_sample_seconds(w, inp, rows)
    secs = [oracle_sample_seconds(w, inp, rows) for _ in range(args.steps)]
    tot = sum(secs)
    value = rows * len(secs) / tot
    sample = (f"first {rows} of the {w.t} rows of the workload per step (about {per_step:.0f} s of oracle work "
              f"each), full oracle (router, CSR, experts), one thread")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(secs) * w.t / rows,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "t": w.t, "h": w.h, "inter": w.inter, "E": w.E,
                                        "k": w.k, "shared_inter": w.shared_inter},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# Our arm
# --------------------------------------------------------------------------

def run_ours(args, w: synth.Workload):
    import torch
    import torch.distributed as dist

    from routed_expert_prefill_gb300 import build as B

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev_name = f"cuda:{local}"
    if rank == 0 or not os.path.exists(os.path.join(ROOT, "routed_expert_prefill_gb300", "libmoe_gb300.so")):
        B.build()
    if world > 1:
        dist.barrier()
    from routed_expert_prefill_gb300 import moe

    inp = synth.make_inputs(w)
    dev = moe.upload_inputs(inp, dev_name)
    dims = moe.dims_of(w.t, w.h, w.inter, w.E, w.k, w.shared_inter)
    flags = args.flags
    ws = moe.new_workspace(dims, flags, dev_name)
    out = torch.empty((w.t, w.h), dtype=torch.bfloat16, device=dev_name)
    stream = torch.cuda.current_stream()
    bufs = dict(route=(torch.empty((w.t, w.k), dtype=torch.int32, device=dev_name),
                       torch.empty((w.t, w.k), dtype=torch.float32, device=dev_name)),
                csr=moe.Csr(torch.empty(w.E + 1, dtype=torch.int32, device=dev_name),
                            torch.empty(w.t * w.k, dtype=torch.int32, device=dev_name),
                            torch.empty(w.t * w.k, dtype=torch.float32, device=dev_name),
                            torch.empty(w.t * w.k, dtype=torch.int32, device=dev_name)))
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev_name)

    def step():
        return moe.moe_forward(dev, dims, flags, ws=ws, out=out, bufs=bufs)

    for _ in range(args.warmup):
        res = step()
    torch.cuda.synchronize()
    status = moe.read_device_status(ws)
    if status != 0:
        raise RuntimeError(f"device-side status {status} after warm-up")
    counts = np.diff(res["csr"].offsets.cpu().numpy())
    work = step_work(w, counts)

    # ---- device-resident timed region (L2 flushed between steps, untimed).
    # The step is captured once into a CUDA graph and replayed, so the
    # timing is the GPU's, not the host's launch rate.
    graph = None
    if not args.no_graph:
        side = torch.cuda.Stream(device=dev_name)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        graph.replay()
        torch.cuda.synchronize()

    def timed(run, n):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for i in range(n):
            flush.fill_(float(i))
            starts[i].record(stream)
            run()
            ends[i].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in zip(starts, ends)]

    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    step_ms = timed(graph.replay if graph is not None else step, args.steps)
    wall = time.perf_counter() - wall0
    # per-kernel device time: the same steps launched directly, each launch
    # bracketed by CUDA events on the launching stream
    moe.profile_enable(True)
    eager_ms = timed(step, args.steps)
    moe.profile_enable(False)
    prof = moe.profile_read()
    clocks = sampler.stop()
    ms = max_over_ranks(sum(step_ms) / len(step_ms), dev_name)
    gpu_launches = sum(v[0] for v in prof.values())

    # ---- end to end through the public API with host buffers: every step
    # copies its chunk of x in from pinned host memory and its block output
    # back.  When the step's weights or its gathered token rows exceed L2,
    # steps run back to back as a serving loop would: two x and two output
    # buffers, the copies on streams of their own overlapping the
    # neighbouring steps' forward passes, one timed region over all K steps.
    # Otherwise (decode-sized steps, whose weights would stay in L2) each
    # step is timed alone on one stream, copies included, with the L2 flush
    # between steps outside the events.
    x_host = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
    out_hosts = [torch.empty((w.t, w.h), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_devs = [torch.empty_like(dev["x"]) for _ in range(2)]
    outs = [out, torch.empty_like(out)]
    s_in, s_out = torch.cuda.Stream(device=dev_name), torch.cuda.Stream(device=dev_name)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # x of the buffer copied in
    ev_done = [torch.cuda.Event() for _ in range(2)]  # forward done: x free, output ready
    ev_out = [torch.cuda.Event() for _ in range(2)]   # output copied back: buffer free
    pipelined = work["bytes"] > L2_BYTES or w.t * (w.k + 1) * w.h * 2 > L2_BYTES

    def e2e_step(i):
        bi = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_done[bi])
            x_devs[bi].copy_(x_host, non_blocking=True)
            ev_in[bi].record(s_in)
        stream.wait_event(ev_in[bi])
        if i >= 2:
            stream.wait_event(ev_out[bi])
        moe.moe_forward(dict(dev, x=x_devs[bi]), dims, flags, ws=ws, out=outs[bi], bufs=bufs)
        ev_done[bi].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[bi])
            out_hosts[bi].copy_(outs[bi], non_blocking=True)
            ev_out[bi].record(s_out)

    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize()
    if pipelined:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for i in range(args.steps):
            e2e_step(i)
        e1.record(s_out)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dev_name)
    else:
        e_starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        e_ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        dev1 = dict(dev, x=x_devs[0])
        for i in range(args.steps):
            flush.fill_(float(i))
            e_starts[i].record(stream)
            x_devs[0].copy_(x_host, non_blocking=True)
            moe.moe_forward(dev1, dims, flags, ws=ws, out=outs[0], bufs=bufs)
            out_hosts[0].copy_(outs[0], non_blocking=True)
            e_ends[i].record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(e_starts, e_ends)) / args.steps, dev_name)
    x_host_bytes, out_host_bytes = int(x_host.numel() * 2), int(out_hosts[0].numel() * 2)

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    # dominant kernel = largest share of device time
    fam_time = {}
    fam_launch = {}
    for name, (n, tms) in prof.items():
        f = kernel_family(name)
        fam_time[f] = fam_time.get(f, 0.0) + tms
        fam_launch[f] = fam_launch.get(f, 0) + n
    dom = max(fam_time, key=fam_time.get)
    per_launch_ms = fam_time[dom] / fam_launch[dom]
    launches_per_step = fam_launch[dom] / args.steps
    kw = work["by_kernel"].get(dom)
    roofline = None
    if kw is not None:
        kb = kw["bytes"] / launches_per_step
        kf = kw["flops"] / launches_per_step
        hbm_t = kb / (peaks["hbm_gbs"] * 1e9)
        ten_t = kf / (peaks["bf16_tflops"] * 1e12)
        if hbm_t >= ten_t:
            ach = kb / (per_launch_ms * 1e-3) / 1e9
            roofline = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": ach / peaks["hbm_gbs"], "traffic": None}
        else:
            ach = kf / (per_launch_ms * 1e-3) / 1e12
            roofline = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                        "frac": ach / peaks["bf16_tflops"], "traffic": None}
        roofline["traffic"] = measured_traffic(w.name, dom, flags)
        roofline.update({"kernel": dom, "peak_source": peak_src,
                         "kernel_ms_per_launch": per_launch_ms,
                         "algorithmic_bytes_per_launch": kb, "algorithmic_flops_per_launch": kf})
    t_star = max(work["flops"] / (peaks["bf16_tflops"] * 1e12), work["bytes"] / (peaks["hbm_gbs"] * 1e9))
    step_bound = "tensor" if work["flops"] / (peaks["bf16_tflops"] * 1e12) > work["bytes"] / (peaks["hbm_gbs"] * 1e9) else "hbm"

    cpu = None
    if not args.no_cpu_baseline:
        # a bounded sample of about 10 s of oracle work
        rows = calibrated_rows(w, inp, 10.0)
        if args.oracle_rows:
            rows = min(rows, args.oracle_rows)
        secs = oracle_sample_seconds(w, inp, rows)
        cpu = {"value": rows / secs, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"first {rows} of {w.t} rows (about 10 s of work), one full oracle pass "
                         f"(router, CSR, experts), 1 thread"}

    value = job_tokens_per_s(world, w.t, ms)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "t": w.t, "h": w.h, "inter": w.inter, "E": w.E, "k": w.k,
                   "shared_inter": w.shared_inter, "flags": flags, "parallelism": f"replicas{world}",
                   "l2": "flushed between timed steps (2x L2 write, untimed); expert weights also exceed L2",
                   "touched_experts": work["touched"], "max_rows_per_expert": work["max_rows"],
                   "step_flops": work["flops"], "step_bytes": work["bytes"],
                   "step_tflops": work["flops"] / (ms * 1e-3) / 1e12,
                   "step_gbs": work["bytes"] / (ms * 1e-3) / 1e9,
                   "step_roofline_frac": t_star / (ms * 1e-3), "step_bound": step_bound,
                   "wall_s_timed_region": wall,
                   "timing": "eager launches" if graph is None else "CUDA graph replay of one captured step",
                   "eager_ms_per_step": sum(eager_ms) / len(eager_ms)},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": job_tokens_per_s(world, w.t, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": x_host_bytes, "d2h_bytes_per_step": out_host_bytes,
                "timing": ("steps back to back, copies overlapping neighbouring steps (step bytes exceed L2)"
                           if pipelined else "each step alone, copies included, L2 flushed between steps")},
        "gpu_launches": gpu_launches,
        "kernels": {k: {"launches": v[0], "ms": v[1]} for k, v in prof.items()},
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--flags", type=int, default=16, help="moe_experts_fwd flags (16: packed weights)")
    ap.add_argument("--no-graph", action="store_true", help="time eager launches instead of graph replays")
    ap.add_argument("--oracle-rows", type=int, default=0, help="cap on the oracle sample's rows (0: time-budgeted)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    w = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()

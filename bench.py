"""Benchmark of the routed-MoE FFN over one prompt chunk on GB300.

A step is one pass of the whole path over one chunk: router top-k, CSR
grouping, and the expert FFNs (shared expert, gate/up + silu*up, down +
weighted scatter-add), i.e. moe_route_csr -> moe_experts_fwd on one stream.
Inputs are synthetic (routed_expert_prefill_gb300.synth) and resident in HBM
for ``value``; ``e2e`` copies x in from pinned host memory and the block
output back every step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--workloads LIST|none] [--impl ours|reference]

The headline workload is t=4096, h=4096, inter=1536, E=256, k=8 (the largest
single-GPU configuration); the same line carries, under ``workloads``, the
skewed t=4096 chunk, the t=512 chunk and the decode-shaped t=1/2/4/8 chunks,
each timed the same way.

Timing: W untimed warm-up steps, then exactly K timed steps, each a replay of
the step captured as a CUDA graph, bracketed by CUDA events on the launching
stream, with a write larger than L2 between steps (outside the events);
``ms_per_step`` is the median.  ``sustained`` repeats the same measurement
for at least one second and 50 runs.

Multi-GPU (torchrun): every rank runs its own chunk (weak scaling, no
collective on the data path); value = all ranks' rows over the max-over-ranks
time.
"""

import os

# Each oracle worker runs single-threaded; the pool spreads rows over cores.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import multiprocessing as mp  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import threading  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from routed_expert_prefill_gb300 import synth  # noqa: E402

METRIC = "prefill tokens/s and % of roofline (tensor or HBM) for routed MoE FFN, 1 GB300"
DEFAULT_WORKLOAD = "t4096_h4096_e256"
EXTRA_WORKLOADS = ("t4096_h2048_e128_skewed", "t512_h2048_e128", "decode_t1_h2048_e128",
                   "decode_t2_h2048_e128", "decode_t4_h2048_e128", "decode_t8_h2048_e128",
                   "t4096_h4096_e256_b2", "t4096_h4096_e256_b3", "t4096_h4096_e256_b8")
# The streamed-experts line: the headline chunk with its routed records in
# host memory, half of them resident in a device pool after the first chunk.
STREAMED = "t4096_h4096_e256_streamed"
STREAMED_MISS2 = "t4096_h4096_e256_streamed_miss2"  # the ring's records from a 2-bit miss store
STREAMED_CFG = dict(pool_slots=128, ring_slots=64, group=8)  # prefill.rs RING and GROUP
L2_BYTES = 129 * 2 ** 20
SUSTAIN_S, SUSTAIN_MIN_RUNS, SUSTAIN_MAX_RUNS = 1.0, 50, 20000
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
MOE_PACKED_WEIGHTS = 0x10


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# --------------------------------------------------------------------------
# Algorithmic work of one step (from the step's actual routing)
# --------------------------------------------------------------------------

def matrix_bytes(rows, K, bits=4):
    """Bytes of one quantised matrix: codes of `bits` bits + fp16 scale and bias per 64."""
    return rows * K * bits // 8 + 2 * 2 * (rows * K // 64)


def record_bytes(h, inter, bits=4):
    """Bytes of one quantised expert record (gate, up, down)."""
    return 3 * matrix_bytes(inter, h, bits)


def step_work(w: synth.Workload, counts: np.ndarray) -> dict:
    touched = int((counts > 0).sum())
    n = int(counts.sum())
    t, h, I, Is, E, k, bits = w.t, w.h, w.inter, w.shared_inter, w.E, w.k, w.bits
    flops = 2 * t * h * E + 6 * n * h * I + 6 * t * h * Is
    wbytes = touched * record_bytes(h, I, bits) + (record_bytes(h, Is, bits) if Is else 0)
    io = 2 * t * h * 2 + E * h * 2 + t * k * 8
    by_kernel = {
        # gate+up weights of touched experts (and the shared expert) + x in + hg out
        "gateup": dict(bytes=touched * 2 * matrix_bytes(I, h, bits)
                       + (2 * matrix_bytes(Is, h, bits) if Is else 0)
                       + t * h * 2 + (n * I + t * Is) * 2,
                       flops=4 * n * h * I + 4 * t * h * Is),
        # down weights + hg in + fp32 block accumulator in/out
        "down": dict(bytes=touched * matrix_bytes(h, I, bits)
                     + (matrix_bytes(h, Is, bits) if Is else 0)
                     + (n * I + t * Is) * 2 + 2 * t * h * 4,
                     flops=2 * n * h * I + 2 * t * h * Is),
        # router (scores + exact refinement): x and router weights in, idx/w out
        "route": dict(bytes=t * h * 2 + E * h * 2 + t * k * 8, flops=2 * t * h * E),
        # the fused decode launch: the whole step
        "decode_fused": dict(bytes=wbytes + io, flops=flops),
    }
    return dict(touched=touched, pairs=n, max_rows=int(counts.max()), flops=flops,
                bytes=wbytes + io, by_kernel=by_kernel)


def step_roofline(work: dict, ms: float, peaks: dict) -> dict:
    """T* = max(F / bf16 peak, B / HBM peak) against the measured step time."""
    tf = work["flops"] / (peaks["bf16_tflops"] * 1e12)
    tb = work["bytes"] / (peaks["hbm_gbs"] * 1e9)
    return {"frac": max(tf, tb) / (ms * 1e-3), "bound": "tensor" if tf > tb else "hbm",
            "t_star_us": 1e6 * max(tf, tb), "tflops": work["flops"] / (ms * 1e-3) / 1e12,
            "gbs": work["bytes"] / (ms * 1e-3) / 1e9}


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of
# the packed expert kernels, from one ncu capture of the bench command on a
# GB300; valid while the kernel sources hash to `src` (reported as null
# otherwise).
PACKED_SOURCES = ("experts_packed.cu", "tc_ptx.cuh", "tc_common.cuh", "common.cuh", "experts.cuh")
MEASURED_TRAFFIC = {
    ("t4096_h4096_e256", "gateup", 16): dict(bytes=2335.95e6, src="86c5aeef4802cbcb"),
    ("t4096_h4096_e256", "down", 16): dict(bytes=1710.03e6, src="86c5aeef4802cbcb"),
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
    for fam in ("gateup", "down", "route", "decode_fused"):
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
        sm, mx, pw, reasons = [], [], [], set()
        for ln in self.lines:
            f = [s.strip() for s in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                pw.append(float(f[3]))
            except ValueError:
                continue
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                                 f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        # "under load": samples drawing more than a third of the peak power seen
        loaded = [s for s, p in zip(sm, pw) if p > max(pw) / 3] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "samples_under_load": len(loaded), "power_w_max": max(pw)}


# --------------------------------------------------------------------------
# The CPU oracle, timed on the host's cores
# --------------------------------------------------------------------------

_POOL_INPUTS = None  # the workload's inputs, set before the pool forks (workers share them)


def _oracle_worker(task):
    """One worker: the oracle as it stands on rows [a, b) of the workload."""
    a, b, k, h, inter, shared_inter = task
    from oracle import moe_oracle as O

    inp = _POOL_INPUTS
    O.moe_forward(dict(inp, x=inp["x"][a:b]), k, h, inter, shared_inter)
    return b - a


class OraclePool:
    """The CPU oracle over a sample of a workload's rows, on every host core.

    A row's output depends on that row alone, so the sample's rows are split
    into one contiguous range per core and each worker runs the unmodified
    oracle (router, grouping, experts) on its range.  The pool forks before
    any CUDA call, so the workers share the inputs without copying them."""

    def __init__(self, w: synth.Workload, inp: dict, cores: int):
        global _POOL_INPUTS
        _POOL_INPUTS = inp
        self.w, self.inp, self.cores = w, inp, cores
        self.pool = mp.get_context("fork").Pool(cores) if cores > 1 else None

    def seconds(self, rows: int) -> float:
        w = self.w
        n = min(self.cores, rows)
        cuts = np.linspace(0, rows, n + 1).astype(int)
        tasks = [(int(cuts[i]), int(cuts[i + 1]), w.k, w.h, w.inter, w.shared_inter) for i in range(n)]
        t0 = time.perf_counter()
        if self.pool is None:
            for tk in tasks:
                _oracle_worker(tk)
        else:
            self.pool.map(_oracle_worker, tasks, chunksize=1)
        return time.perf_counter() - t0

    def rows_for(self, budget_s: float) -> int:
        """Rows whose pass takes about budget_s (from a timed probe of two rows per core)."""
        probe = min(self.w.t, 2 * self.cores)
        s = self.seconds(probe)
        return int(max(probe, min(self.w.t, probe * budget_s / max(s, 1e-9))))

    def close(self):
        if self.pool is not None:
            self.pool.close()
            self.pool.join()


def oracle_one_core_seconds(w: synth.Workload, inp: dict, rows: int) -> float:
    from oracle import moe_oracle as O

    t0 = time.perf_counter()
    O.moe_forward(dict(inp, x=inp["x"][:rows]), w.k, w.h, w.inter, w.shared_inter)
    return time.perf_counter() - t0


def cpu_baseline(pool: OraclePool, w: synth.Workload, inp: dict, budget_s: float, one_core: bool) -> dict:
    rows = pool.rows_for(budget_s)
    secs = pool.seconds(rows)
    res = {"value": rows / secs, "unit": "tokens/s", "cores": pool.cores, "kind": "oracle",
           "sample": f"first {rows} of the {w.t} rows, split over {pool.cores} host cores (one oracle "
                     f"process per core: router, grouping, experts in fp64), {secs:.1f} s"}
    if one_core:
        probe = min(w.t, 4)
        per_row = oracle_one_core_seconds(w, inp, probe) / probe
        r1 = int(max(probe, min(w.t, budget_s / max(per_row, 1e-9))))
        s1 = oracle_one_core_seconds(w, inp, r1)
        res["one_core"] = {"value": r1 / s1, "unit": "tokens/s", "cores": 1,
                           "sample": f"first {r1} of the {w.t} rows on one core, {s1:.1f} s"}
    return res


def run_reference(args, w: synth.Workload):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    inp = synth.make_inputs(w)
    pool = OraclePool(w, inp, host_cores())
    try:
        # each step a bounded sample: the whole run stays within about 150 s
        per_step = min(10.0, 150.0 / max(1, args.steps + args.warmup))
        rows = pool.rows_for(per_step)
        if args.oracle_rows:
            rows = min(rows, args.oracle_rows)
        for _ in range(args.warmup):
            pool.seconds(rows)
        secs = [pool.seconds(rows) for _ in range(args.steps)]
    finally:
        pool.close()
    mean_s = sum(secs) / len(secs)
    value = rows / mean_s
    sample = (f"first {rows} of the {w.t} rows of the workload per step, split over {pool.cores} host cores "
              f"(one oracle process per core: router, grouping, experts in fp64)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * mean_s,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "t": w.t, "h": w.h, "inter": w.inter, "E": w.E,
                                        "k": w.k, "shared_inter": w.shared_inter, "rows_per_step": rows,
                                        "step": f"the oracle over {rows} of the {w.t} rows"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": pool.cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# Our arm
# --------------------------------------------------------------------------

class Ctx:
    """Per-process state of our arm: torch, the binding, ranks, device buffers."""

    def __init__(self, args):
        import torch
        import torch.distributed as dist

        from routed_expert_prefill_gb300 import build as B

        self.torch, self.dist, self.args = torch, dist, args
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        if self.world > 1:
            dist.init_process_group("nccl")
        torch.cuda.set_device(self.local)
        self.dev = f"cuda:{self.local}"
        if self.rank == 0 or not os.path.exists(os.path.join(ROOT, "routed_expert_prefill_gb300",
                                                             "libmoe_gb300.so")):
            B.build()
        self.barrier()
        from routed_expert_prefill_gb300 import moe

        self.moe = moe
        self.flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=self.dev)
        self.weights = {}  # device weights per weight recipe (the decode workloads share one)

    def barrier(self):
        if self.world > 1:
            self.dist.barrier()

    def device_inputs(self, w: synth.Workload, inp: dict, flags: int) -> dict:
        moe, torch = self.moe, self.torch
        key = (w.h, w.inter, w.E, w.shared_inter, w.seed, w.skew, w.shared_gate, w.bits)
        if key not in self.weights:
            self.weights.clear()
            torch.cuda.empty_cache()
            dev = moe.upload_inputs(inp, self.dev)
            if flags & MOE_PACKED_WEIGHTS:
                moe.add_packed(dev, moe.dims_of(w.t, w.h, w.inter, w.E, w.k, w.shared_inter, w.bits))
            self.weights[key] = dev
        dev = dict(self.weights[key])
        dev["x"] = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).to(self.dev)
        return dev


def measure(ctx: Ctx, w: synth.Workload, inp: dict, headline: bool) -> dict:
    """Time one workload: graph-replayed steps (value), per-kernel events, the
    sustained run, and the end-to-end loop through the public API."""
    torch, moe, args = ctx.torch, ctx.moe, ctx.args
    flags = args.flags
    dev = ctx.device_inputs(w, inp, flags)
    dims = moe.dims_of(w.t, w.h, w.inter, w.E, w.k, w.shared_inter, w.bits)
    ws = moe.new_workspace(dims, flags, ctx.dev)
    out = torch.empty((w.t, w.h), dtype=torch.bfloat16, device=ctx.dev)
    stream = torch.cuda.current_stream()
    bufs = dict(route=(torch.empty((w.t, w.k), dtype=torch.int32, device=ctx.dev),
                       torch.empty((w.t, w.k), dtype=torch.float32, device=ctx.dev)),
                csr=moe.Csr(torch.empty(w.E + 1, dtype=torch.int32, device=ctx.dev),
                            torch.empty(w.t * w.k, dtype=torch.int32, device=ctx.dev),
                            torch.empty(w.t * w.k, dtype=torch.float32, device=ctx.dev),
                            torch.empty(w.t * w.k, dtype=torch.int32, device=ctx.dev)))
    flush = ctx.flush

    def step():
        return moe.moe_forward(dev, dims, flags, ws=ws, out=out, bufs=bufs)

    for _ in range(args.warmup):
        res = step()
    torch.cuda.synchronize()
    status = moe.read_device_status(ws)
    if status != 0:
        raise RuntimeError(f"{w.name}: device-side status {status} after warm-up")
    counts = np.diff(res["csr"].offsets.cpu().numpy())
    work = step_work(w, counts)

    # ---- device-resident timed region: the step captured once into a CUDA
    # graph and replayed, so the timing is the GPU's, not the host's launch
    # rate; L2 flushed between steps, outside the events.
    graph = None
    if not args.no_graph:
        side = torch.cuda.Stream(device=ctx.dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        graph.replay()
        torch.cuda.synchronize()
    run = graph.replay if graph is not None else step

    def timed(fn, n):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for i in range(n):
            flush.fill_(float(i))
            starts[i].record(stream)
            fn()
            ends[i].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in zip(starts, ends)]

    sampler = ClockSampler(ctx.local)
    ctx.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    step_ms = timed(run, args.steps)
    wall = time.perf_counter() - wall0
    ms = max_over_ranks(statistics.median(step_ms), ctx.dev)

    # sustained: the same measurement repeated for >= 1 s and >= 50 runs
    sustained = None
    if not args.no_sustain:
        per = statistics.median(step_ms) + 0.05  # + the flush
        n = int(min(SUSTAIN_MAX_RUNS, max(SUSTAIN_MIN_RUNS, 1.0 + SUSTAIN_S * 1e3 / per)))
        s0 = time.perf_counter()
        sus_ms = timed(run, n)
        sus_wall = time.perf_counter() - s0
        sustained = {"runs": n, "median_ms": statistics.median(sus_ms), "mean_ms": sum(sus_ms) / n,
                     "p10_ms": float(np.percentile(sus_ms, 10)), "p90_ms": float(np.percentile(sus_ms, 90)),
                     "wall_s": sus_wall, "device_s": sum(sus_ms) / 1e3}
    clocks = sampler.stop()

    # per-kernel device time: the same steps launched directly, each launch
    # bracketed by CUDA events on the launching stream
    moe.profile_enable(True)
    eager_ms = timed(step, args.steps)
    moe.profile_enable(False)
    prof = moe.profile_read()
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
    s_in, s_out = torch.cuda.Stream(device=ctx.dev), torch.cuda.Stream(device=ctx.dev)
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
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, ctx.dev)
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
        e2e_ms = max_over_ranks(statistics.median(s.elapsed_time(e) for s, e in zip(e_starts, e_ends)), ctx.dev)
    if moe.read_device_status(ws) != 0:
        raise RuntimeError(f"{w.name}: device-side status set during the timed runs")

    peaks, peak_src = load_peaks()
    fam_time, fam_launch = {}, {}
    for name, (n, tms) in prof.items():
        f = kernel_family(name)
        fam_time[f] = fam_time.get(f, 0.0) + tms
        fam_launch[f] = fam_launch.get(f, 0) + n
    dom = max(fam_time, key=fam_time.get)  # the dominant kernel: largest share of device time
    per_launch_ms = fam_time[dom] / fam_launch[dom]
    launches_per_step = fam_launch[dom] / args.steps
    kw = work["by_kernel"].get(dom)
    roofline = None
    if kw is not None:
        kb = kw["bytes"] / launches_per_step
        kf = kw["flops"] / launches_per_step
        if kb / (peaks["hbm_gbs"] * 1e9) >= kf / (peaks["bf16_tflops"] * 1e12):
            ach = kb / (per_launch_ms * 1e-3) / 1e9
            roofline = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": ach / peaks["hbm_gbs"]}
        else:
            ach = kf / (per_launch_ms * 1e-3) / 1e12
            roofline = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                        "frac": ach / peaks["bf16_tflops"]}
        roofline.update({"traffic": measured_traffic(w.name, dom, flags), "kernel": dom,
                         "peak_source": peak_src + " (burst)", "kernel_ms_per_launch": per_launch_ms,
                         "kernel_share_of_step": fam_time[dom] / sum(fam_time.values()),
                         "algorithmic_bytes_per_launch": kb, "algorithmic_flops_per_launch": kf})
    sr = step_roofline(work, ms, peaks)
    return dict(
        name=w.name, value=job_tokens_per_s(ctx.world, w.t, ms), ms=ms, step_ms=step_ms, wall=wall,
        work=work, step_roofline=sr, roofline=roofline, sustained=sustained, clocks=clocks,
        eager_ms=statistics.median(eager_ms), gpu_launches=gpu_launches,
        kernels={k: {"launches": v[0], "ms": v[1]} for k, v in prof.items()},
        e2e={"value": job_tokens_per_s(ctx.world, w.t, e2e_ms), "unit": "tokens/s",
             "h2d_bytes_per_step": int(x_host.numel() * 2), "d2h_bytes_per_step": int(out_hosts[0].numel() * 2),
             "timing": ("steps back to back, copies overlapping neighbouring steps (step bytes exceed L2)"
                        if pipelined else "each step alone, copies included, L2 flushed between steps; median")},
        graph=graph is not None, flags=flags)


def measure_streamed(ctx: Ctx, w: synth.Workload, inp: dict, miss_bits: int = 0) -> dict:
    """Time moe_forward_streamed on workload ``w`` in its steady state (the
    pool filled by the warm-up chunks): every step routes, plans, fetches the
    non-resident records from pinned host memory over the host link and runs
    the batches.  With ``miss_bits`` the ring's records come from a store
    packed at that width (the workload's records drawn at that width).
    Bound: the host-to-device copy rate, measured here on the same pinned
    buffer."""
    torch, moe, args = ctx.torch, ctx.moe, ctx.args
    flags = MOE_PACKED_WEIGHTS
    host_miss = None
    if miss_bits:
        wm = w.replace(bits=miss_bits)
        dm = ctx.device_inputs(wm, synth.make_inputs(wm), flags)
        host_miss = dm["packed"].cpu().pin_memory()
        del dm
    dev = ctx.device_inputs(w, inp, flags)
    dims = moe.dims_of(w.t, w.h, w.inter, w.E, w.k, w.shared_inter, w.bits)
    host = dev["packed"].cpu().pin_memory()
    st = moe.Streamer(dims, STREAMED_CFG["pool_slots"], STREAMED_CFG["ring_slots"], STREAMED_CFG["group"], host,
                      ctx.dev, host_miss_records=host_miss, miss_bits=miss_bits)
    ws = moe.new_workspace(dims, flags, ctx.dev)
    out = torch.empty((w.t, w.h), dtype=torch.bfloat16, device=ctx.dev)
    bufs = dict(route=(torch.empty((w.t, w.k), dtype=torch.int32, device=ctx.dev),
                       torch.empty((w.t, w.k), dtype=torch.float32, device=ctx.dev)),
                csr=moe.Csr(torch.empty(w.E + 1, dtype=torch.int32, device=ctx.dev),
                            torch.empty(w.t * w.k, dtype=torch.int32, device=ctx.dev),
                            torch.empty(w.t * w.k, dtype=torch.float32, device=ctx.dev),
                            torch.empty(w.t * w.k, dtype=torch.int32, device=ctx.dev)))
    stream = torch.cuda.current_stream()

    def step():
        return moe.moe_forward_streamed(dev, dims, st, flags, ws=ws, out=out, bufs=bufs)

    for _ in range(args.warmup):
        res = step()
    torch.cuda.synchronize()
    if moe.read_device_status(ws) != 0:
        raise RuntimeError(f"{STREAMED}: device-side status after warm-up")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    stats = []
    for i in range(args.steps):
        ctx.flush.fill_(float(i))
        starts[i].record(stream)
        res = step()
        ends[i].record(stream)
        stats.append(res["stats"])
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ms = max_over_ranks(statistics.median(step_ms), ctx.dev)
    moe.profile_enable(True)
    for _ in range(3):
        step()
    moe.profile_enable(False)
    prof = moe.profile_read()
    kernel_ms = sum(v[1] for v in prof.values()) / 3
    if moe.read_device_status(ws) != 0:
        raise RuntimeError(f"{STREAMED}: device-side status set during the timed runs")
    st.close()
    # the host-to-device copy rate of this pinned buffer: 1 GiB, best of 3
    n = min(1 << 30, host.numel())
    dst = torch.empty(n, dtype=torch.uint8, device=ctx.dev)
    rates = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dst.copy_(host[:n], non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        rates.append(n / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    del dst
    h2d_gbs = max(rates)
    last = stats[-1]
    moved = last["bytes"]
    ach = moved / (ms * 1e-3) / 1e9
    return dict(
        value=job_tokens_per_s(ctx.world, w.t, ms), unit="tokens/s", ms_per_step=ms,
        config={"workload": STREAMED_MISS2 if miss_bits else STREAMED, "t": w.t, "h": w.h, "inter": w.inter,
                "E": w.E, "k": w.k, "shared_inter": w.shared_inter, "bits": w.bits, **STREAMED_CFG,
                "miss_bits": miss_bits or w.bits,
                "records": "packed routed records in pinned host memory; shared record on the device"
                           + ("; ring records from a 2-bit miss store" if miss_bits else ""),
                "resident_experts": last["resident"], "filled_per_step": last["filled"],
                "streamed_per_step": last["streamed"], "fetch_batches": last["batches"],
                "bytes_copied_per_step": moved, "step_ms_min": min(step_ms), "step_ms_max": max(step_ms),
                "kernel_ms_per_step": kernel_ms,
                "timing": "median of the K steps, CUDA events around each call (the call waits once "
                          "for the routing on the host); L2 flushed between steps"},
        roofline={"bound": "h2d", "achieved": ach, "peak": h2d_gbs, "unit": "GB/s", "frac": ach / h2d_gbs,
                  "traffic": None, "peak_source": "1 GiB host-to-device copy from the same pinned buffer, "
                                                  "measured in this run (best of 3)"},
        gpu_launches=sum(v[0] for v in prof.values()) // 3,
        kernels={k: {"launches": v[0], "ms": v[1]} for k, v in prof.items()})


def workload_config(w: synth.Workload, m: dict) -> dict:
    work, sr = m["work"], m["step_roofline"]
    return {"workload": w.name, "t": w.t, "h": w.h, "inter": w.inter, "E": w.E, "k": w.k,
            "shared_inter": w.shared_inter, "bits": w.bits,
            "routing": "Zipf-skewed" if w.skew else "near-uniform",
            "flags": m["flags"], "touched_experts": work["touched"], "max_rows_per_expert": work["max_rows"],
            "step_flops": work["flops"], "step_bytes": work["bytes"], "step_tflops": sr["tflops"],
            "step_gbs": sr["gbs"], "step_roofline_frac": sr["frac"], "step_bound": sr["bound"],
            "step_t_star_us": sr["t_star_us"]}


def run_ours(args, w: synth.Workload, pool):
    ctx = Ctx(args)
    inp = pool.inp if pool is not None else synth.make_inputs(w)
    m = measure(ctx, w, inp, True)
    extras = {}
    for name, mb in ((STREAMED, 0), (STREAMED_MISS2, 2)):
        if name in args.extra:
            extras[name] = measure_streamed(ctx, synth.WORKLOADS[DEFAULT_WORKLOAD],
                                            inp if w.name == DEFAULT_WORKLOAD else
                                            synth.make_inputs(synth.WORKLOADS[DEFAULT_WORKLOAD]), mb)
    for name in args.extra:
        if name in (STREAMED, STREAMED_MISS2):
            continue
        wx = synth.WORKLOADS[name]
        mx = measure(ctx, wx, synth.make_inputs(wx), False)
        extras[name] = dict(
            value=mx["value"], unit="tokens/s", ms_per_step=mx["ms"], config=workload_config(wx, mx),
            roofline=mx["roofline"], e2e=mx["e2e"], gpu_launches=mx["gpu_launches"],
            sustained=mx["sustained"], clocks=mx["clocks"],
            kernels=mx["kernels"])
    if ctx.rank != 0:
        ctx.barrier()
        if ctx.world > 1:
            ctx.dist.destroy_process_group()
        return

    cpu = None
    if pool is not None:
        cpu = cpu_baseline(pool, w, inp, 10.0, one_core=w.t * w.h * w.inter <= 512 * 2048 * 768)
        pool.close()

    cfg = workload_config(w, m)
    cfg.update({"parallelism": f"replicas{ctx.world}",
                "l2": "flushed between timed steps (2x L2 write, untimed); expert weights also exceed L2",
                "timing": ("median of the K timed steps, each a CUDA graph replay of one captured step"
                           if m["graph"] else "median of the K timed steps, eager launches"),
                "wall_s_timed_region": m["wall"], "eager_ms_per_step": m["eager_ms"],
                "step_ms_min": min(m["step_ms"]), "step_ms_max": max(m["step_ms"])})
    line = {
        "metric": METRIC, "value": m["value"], "unit": "tokens/s", "n_gpus": ctx.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": m["ms"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": cfg,
        "step_roofline_frac": m["step_roofline"]["frac"],
        "roofline": m["roofline"],
        "cpu_baseline": cpu,
        "e2e": m["e2e"],
        "gpu_launches": m["gpu_launches"],
        "sustained": m["sustained"],
        "kernels": m["kernels"],
        "clocks": m["clocks"],
        "workloads": extras,
    }
    print(json.dumps(line), flush=True)
    ctx.barrier()
    if ctx.world > 1:
        ctx.dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--workloads", default="default",
                    help="extra workloads timed in the same run: comma list, 'none', or 'default' "
                         "(the other benchmark workloads when the headline one is timed)")
    ap.add_argument("--flags", type=int, default=MOE_PACKED_WEIGHTS, help="moe_experts_fwd flags (16: packed weights)")
    ap.add_argument("--no-graph", action="store_true", help="time eager launches instead of graph replays")
    ap.add_argument("--no-sustain", action="store_true", help="skip the >= 1 s sustained measurement")
    ap.add_argument("--oracle-rows", type=int, default=0, help="cap on the oracle sample's rows (0: time-budgeted)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.impl == "ours" and args.warmup < 3:
        ap.error("--warmup must be at least 3")
    w = synth.WORKLOADS[args.workload]
    if args.workloads == "default":
        args.extra = ([STREAMED, STREAMED_MISS2] + [n for n in EXTRA_WORKLOADS if n != w.name]
                      if w.name == DEFAULT_WORKLOAD else [])
    elif args.workloads == "none":
        args.extra = []
    else:
        args.extra = [n for n in args.workloads.split(",") if n]
        for n in args.extra:
            if n not in synth.WORKLOADS and n not in (STREAMED, STREAMED_MISS2):
                ap.error(f"unknown workload {n}")
    if args.impl == "reference":
        run_reference(args, w)
        return
    # the oracle pool forks before any CUDA call (rank 0 of a 1-GPU run only)
    pool = None
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if not args.no_cpu_baseline and world == 1:
        pool = OraclePool(w, synth.make_inputs(w), host_cores())
    run_ours(args, w, pool)


if __name__ == "__main__":
    main()

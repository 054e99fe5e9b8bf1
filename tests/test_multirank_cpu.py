"""Multi-rank host logic of bench.py on CPU: two gloo ranks, no GPU.

Each rank runs its own chunk (weak scaling, no collective on the data path);
the timed interval is the maximum over ranks and the job's throughput counts
every rank's rows.
"""

import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        ms = bench.max_over_ranks(1.5 + rank, "cpu")  # rank 1 is the slow one
        out[rank] = (ms, bench.job_tokens_per_s(world, 512, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    world = 2
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1]
    ms, tps = out[0]
    assert ms == 2.5
    assert tps == pytest.approx(2 * 512 / 2.5e-3)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.25, "cpu") == 3.25
    assert bench.job_tokens_per_s(1, 4096, 1.0) == 4096e3

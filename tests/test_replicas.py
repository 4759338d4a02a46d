"""The multi-process path of bench.py on CPU: two gloo ranks (world size 2)
run the same host logic the benchmark runs under torchrun on N GPUs --
barrier, max-over-ranks timing and the weak-scaling replica throughput --
with no GPU.  Replicas only: every rank processes the whole per-GPU
workload, so no collective touches the data path."""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier(world)
        ms = 10.0 + 5.0 * rank  # rank 1 is the slower one
        worst = bench.max_over_ranks(ms, world)
        value = bench.replica_rows_per_s(12288, 20, world, worst)
        bench.barrier(world)
        q.put((rank, worst, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_by_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0, f"rank process exited with {p.exitcode}"
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, worst, value in got:
        assert worst == 15.0  # every rank reports the slowest rank's time
        assert value == pytest.approx(12288 * 20 * 2 / 15e-3)


def test_single_rank_is_the_plain_rate():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.replica_rows_per_s(4096, 10, 1, 2.0) == pytest.approx(4096 * 10 / 2e-3)

"""The multi-GPU bench path on CPU: two `gloo` ranks agree on the slowest
rank's time, and the whole-job throughput counts every rank's bytes.

On GPUs the bench runs one independent replica of the workload per rank
(the path has no exchange step); only the timing is reduced across ranks.
"""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank            # rank 1 is the slow one
        q.put((rank, bench.max_over_ranks(mine)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=5) for _ in range(world))
    assert got == {0: 15.0, 1: 15.0}


def test_single_process_and_throughput_formula():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    # 2 ranks x 29,378,560 B x 1000 steps in 10 ms = 5.8757 TB/s
    assert bench.job_tbps(2, 29_378_560, 1000, 10.0) == pytest.approx(5.875712)

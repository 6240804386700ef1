"""The multi-rank host logic of bench.py on CPU: two gloo ranks.

bench.py runs one replica of the layer per GPU (the path does not shard), and
reports the whole job's throughput from the slowest rank: every rank waits at
the barrier, and the timed milliseconds are the maximum over ranks.  These
tests run that logic in two CPU processes over the gloo backend.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # a rank's own time: rank 1 is the slow one
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank, world)
        bench.barrier(world)
        q.put((rank, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = {}
    try:
        for _ in range(2):
            rank, v = q.get(timeout=120)
            got[rank] = v
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    assert got == {0: 15.0, 1: 15.0}


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)   # a no-op without a process group

"""The multi-rank host logic of bench.py (replicas, max over ranks) on two
gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        slowest = bench.max_over_ranks(1.0 + rank, world)
        tok_s = bench.aggregate(128, 10, 0.5 + 0.25 * rank, world)
        q.put((rank, slowest, tok_s))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, slowest, tok_s in res:
        assert slowest == 2.0
        # 2 ranks x 10 steps x 128 tokens over the slowest rank's 0.75 s
        assert tok_s == pytest.approx(2 * 10 * 128 / 0.75)


def test_single_rank_needs_no_process_group():
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.aggregate(128, 10, 0.5, 1) == pytest.approx(2560.0)

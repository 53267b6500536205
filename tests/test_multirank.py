"""Replica scaling, host side: two gloo ranks on the CPU.

The forward pass shards by (batch, head) with no exchange, so N GPUs run N
replicas of the workload; the benchmark takes the slowest rank's time and
counts the work of every rank.  These tests run that reduction with
world_size 2 over gloo on 127.0.0.1.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 100.0 + 50.0 * rank          # rank 1 is the slow one
        t = bench.slowest_rank_ms(local_ms, world)
        v = bench.job_throughput(2e12, 10, t, world)
        out[rank] = (t, v)
    finally:
        dist.destroy_process_group()


def test_two_rank_reduction_takes_the_slowest_rank():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        t, v = out[r]
        assert t == pytest.approx(150.0)
        # 2 ranks x 10 steps x 2e12 flops in 0.15 s
        assert v == pytest.approx(2 * 10 * 2e12 / 0.15 / 1e12)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.slowest_rank_ms(12.5, 1) == 12.5
    assert bench.job_throughput(1e12, 4, 2.0, 1) == pytest.approx(2000.0)

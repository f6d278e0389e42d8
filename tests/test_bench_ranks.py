"""The bench's replica aggregation across ranks, on CPU with two gloo ranks: the job time is the
slowest rank's, and the job rate counts every rank's products."""
import os
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks([0.75, 1.25][rank], world, device="cpu")
        out[rank] = (t, bench.job_rate(1_000_000_000, 4, world, t))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = 29500 + os.getpid() % 1000
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        t, rate = res[r]
        assert t == 1.25
        assert rate == pytest.approx(2.0 * 1e9 * 4 * 2 / 1.25 / 1e9)


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.5, 1) == 0.5
    assert bench.job_rate(10**9, 2, 1, 1.0) == 4.0

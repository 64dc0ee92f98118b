"""The N > 1 host path of bench.py with two gloo ranks on the CPU.

Each rank runs an independent replica (the (batch, head) pairs share nothing), so the
only cross-rank logic is the max of the step times and the whole-job throughput.
"""
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        ms = 10.0 + 3.0 * rank                     # rank 1 is the slow one
        worst = bench.max_over_ranks(ms, world, "cpu")
        value = bench.job_throughput(1000, world, worst)
        seeds = [None] * world
        dist.all_gather_object(seeds, bench.rank_seed(rank))
        out[rank] = (worst, value, tuple(seeds))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_throughput():
    world, port = 2, _free_port()
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        worst, value, seeds = res[rank]
        assert worst == 13.0                       # every rank sees the slowest time
        assert abs(value - 2 * 1000 / 0.013) < 1e-6
        assert len(set(seeds)) == world            # replicas draw different inputs


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5, 1, "cpu") == 7.5
    assert bench.job_throughput(10, 1, 1000.0) == 10.0

"""The N > 1 path of bench.py (replicas, one per GPU; rows shard with no
data-path collective): the timing reduction and the whole-job value, run as two
gloo ranks on the CPU, and the reference arm's rule that only rank 0 works."""
import argparse
import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (r + 1) ms for the step and 10 * (r + 1) ms end to end
        ms, e2e = bench.max_over_ranks([1.0 + rank, 10.0 * (1 + rank)])
        dist.barrier()
        out[rank] = (ms, e2e, bench.job_value(world, 4e9, ms))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_and_count_every_replica():
    world, port = 2, 29500 + os.getpid() % 1000
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        ms, e2e, value = out[r]
        assert ms == 2.0 and e2e == 20.0          # the slowest rank's times, on every rank
        assert value == pytest.approx(2 * 4e9 / 2e-3 / 1e9)   # both replicas' bytes


def test_reference_arm_only_rank0_works():
    sys.path.insert(0, ROOT)
    import bench
    args = argparse.Namespace(steps=1, warmup=3)
    assert bench.run_reference(args, rank=1, world=2) is None

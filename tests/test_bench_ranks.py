"""Multi-rank host logic of bench.py on CPU: two gloo ranks, no GPU.

Under torchrun every rank times its own replica of the workload; the job's time is the
slowest rank's, and the job's throughput counts the work of every rank.  The reference arm
runs on rank 0 only.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        # Rank r reports step time 10 + r and layer times that peak on different ranks.
        mine = [10.0 + rank, 3.0 - rank, 1.0 + 2.0 * rank]
        out[rank] = bench.max_over_ranks(mine, "cpu", world)

        class A:
            steps, warmup, workload = 1, 3, "tiny_1d_f32"
        # The reference arm does no work on ranks other than 0.
        if rank != 0:
            out[world + rank] = bench.run_reference(A, rank, world)
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    expect = [11.0, 3.0, 3.0]
    for r in range(world):
        assert out[r] == pytest.approx(expect)
    assert out[world + 1] is None


def test_aggregate_rate_counts_every_rank():
    # 2 ranks, each 1e9 FLOP in 1 ms -> 2e12 FLOP/s = 2000 GFLOP/s.
    assert bench.aggregate_rate(2, 1e9, 1.0) == pytest.approx(2000.0)
    assert bench.aggregate_rate(1, 5e8, 0.5) == pytest.approx(1000.0)

"""The N > 1 plumbing of bench.py, on the CPU with two gloo ranks.

bench.py runs one replica of the hot path per rank (the path partitions by
token: weak scaling, no data-path collective). What is shared is the timing:
every rank's totals are reduced with a maximum, so the slowest rank sets the
job time, and the job rate counts the units of all ranks. The reference arm
runs on rank 0 only; other ranks return without work.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r's per-quantity totals; rank 1 is slower on the first two, rank 0 on the last
        mine = [10.0 + rank, 2.0 + 3 * rank, 7.0 - rank, float(rank)]
        got = bench.max_over_ranks(mine, world, "cpu")
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    expect = [11.0, 5.0, 7.0, 1.0]
    assert res[0] == expect and res[1] == expect


def test_max_over_ranks_single_rank_is_identity():
    assert bench.max_over_ranks([3.0, 1.5], 1) == [3.0, 1.5]


def test_job_rate_counts_all_ranks():
    # 256 tokens per rank in 0.1 ms on each of 4 ranks: 4 * 256 / 1e-4 tokens/s
    assert bench.job_rate(4, 256, 1e-4) == pytest.approx(1.024e7)
    assert bench.job_rate(1, 256, 1e-4) == pytest.approx(2.56e6)


def test_reference_arm_runs_on_rank_zero_only():
    class A:
        steps, warmup, cpu_seconds = 1, 0, 0.1
    assert bench.run_reference(A(), 1, 2) is None

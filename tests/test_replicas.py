"""The benchmark's multi-GPU mode runs independent replicas of the layer (its one-GPU path has no exchange
step); the ranks meet only for the max-over-ranks time.  That host logic, on two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    slowest = bench.max_over_ranks(times[rank])
    value = bench.job_throughput(world, 30, 4096, slowest)
    dist.barrier()
    results[rank] = (slowest, value)
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    times = [12.5, 17.25]  # summed step times (ms) of the two ranks
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(2, port, times, results), nprocs=2, join=True)
        got = dict(results)
    for rank in (0, 1):
        slowest, value = got[rank]
        assert slowest == 17.25
        assert value == pytest.approx(2 * 30 * 4096 / 17.25e-3)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(1, 10, 100, 1.0) == pytest.approx(1e6)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    """Under torchrun the CPU baseline (the oracle) is timed once, by rank 0; other ranks exit quietly."""
    sys.path.insert(0, ROOT)
    import argparse

    import bench

    args = argparse.Namespace(workload="tiny_fp32", steps=1, warmup=0, cpu_seconds=0.1, gpus=2)
    bench.run_reference(args, rank=1)
    assert capsys.readouterr().out == ""

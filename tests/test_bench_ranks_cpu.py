"""The bench's multi-rank path on CPU: two gloo ranks, each timing its own
replica, meet at the barriers; every rank gets the slowest rank's time and
the job throughput counts the units of all ranks.  (The layer has no
exchange step, so this host logic is the whole N > 1 path.)"""

from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.rank_barrier(world)
        ms = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
        bench.rank_barrier(world)
        out[rank] = (ms, bench.job_throughput(1000, world, ms))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(10.0, 12.5), (7.0, 3.0)])
def test_two_gloo_ranks_take_the_slowest_time_and_count_all_units(times):
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, _free_port(), list(times), out), nprocs=world, join=True,
                       start_method="spawn")
    slowest = max(times)
    for rank in range(world):
        ms, value = out[rank]
        assert ms == slowest
        assert value == pytest.approx(1000 * world / (slowest / 1e3))


def test_single_rank_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(4.25, 1, torch.device("cpu")) == 4.25
    assert bench.job_throughput(500, 1, 2.0) == pytest.approx(250000.0)
    bench.rank_barrier(1)  # no process group: a no-op


def test_reference_arm_runs_on_rank_zero_only(capsys):
    """Under torchrun the oracle arm runs and prints on rank 0 alone; the other
    ranks exit without work."""
    import bench

    class A:
        steps, warmup = 1, 0

    assert bench.run_reference(A(), 1, 2) is None
    assert capsys.readouterr().out == ""

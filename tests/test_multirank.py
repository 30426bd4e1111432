"""The benchmark's multi-rank host logic with two gloo ranks on the CPU (no GPU): every rank runs its
own replica, the job's time is the slowest rank's, and the throughput counts the units of all ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r "measured" (10 + r, 4 + 2 r, 6 - r) ms for (step, fwd, bwd)
        vals = bench.max_over_ranks([10.0 + rank, 4.0 + 2 * rank, 6.0 - rank], world, torch.device("cpu"))
        dist.barrier()
        out[rank] = vals + [bench.job_rate(1000, world, vals[0])]
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    assert sorted(res) == [0, 1]
    for r in (0, 1):
        step, fwd, bwd, rate = res[r]
        assert (step, fwd, bwd) == (11.0, 6.0, 6.0)  # element-wise maxima over the ranks
        assert rate == pytest.approx(2 * 1000 / 0.011)  # both replicas' units over the slowest time


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks([1.5, 2.5], 1, torch.device("cpu")) == [1.5, 2.5]
    assert bench.job_rate(500, 1, 2.0) == pytest.approx(250000.0)

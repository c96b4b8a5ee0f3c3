"""The N > 1 host logic of bench.py on CPU: two gloo ranks (no GPU).

Every rank runs an independent replica of the layer (tokens shard with no exchange,
per-token scales are local), so the only cross-rank steps are the barrier around the
timed region and the max over ranks of the step time; the job's rate is all ranks'
units over the slowest rank's time (weak scaling).
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        local_ms = 1.0 + 0.5 * rank                     # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms, world)
        bench.barrier(world)
        out[rank] = (ms, bench.job_rate(2.0e12, world, ms))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_rate():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as man:
        out = man.dict()
        mp.start_processes(rank_main, args=(world, free_port(), out), nprocs=world, join=True, start_method="spawn")
        res = dict(out)
    assert sorted(res) == [0, 1]
    for ms, rate in res.values():
        assert ms == 1.5                                  # the max, seen by every rank
        assert rate == pytest.approx(2.0e12 * 2 / 1.5e-3 / 1e12)   # both ranks' work over the slowest time


def test_single_rank_needs_no_process_group():
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)
    assert bench.job_rate(1.0e12, 1, 2.0) == pytest.approx(500.0)

"""Multi-rank host logic of bench.py on CPU: two gloo ranks agree on the
slowest step time, and the whole-job value counts every rank's queries."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [1.25, 3.5][rank]
        slowest = bench.max_over_ranks(ms, dist, torch.device("cpu"))
        out[rank] = slowest
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_step():
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    assert out[0] == out[1] == 3.5
    # 2 ranks x 64 queries in 3.5 ms
    assert bench.job_value(2, 64, 3.5) == pytest.approx(2 * 64 / 3.5e-3)


def test_single_rank_is_unchanged():
    assert bench.max_over_ranks(2.0, None, None) == 2.0

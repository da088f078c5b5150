"""The bench's multi-GPU path is independent replicas (no data-path
collective): each rank runs the whole layer on its own batch, and the job
is timed by the slowest rank.  These checks run that host logic on two CPU
ranks over gloo."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench._dist()
        assert (ws, r, local) == (world, rank, rank)
        # each replica's own step time; the job is as slow as the slowest
        ms = bench.max_over_ranks(10.0 + 5.0 * rank)
        rate = bench.whole_job_rate(ws, 8192, 20, ms)
        dist.barrier()
        out[rank] = (ms, rate)
    finally:
        dist.destroy_process_group()


def test_two_replicas_time_and_rate():
    world = 2
    with mp.get_context("spawn").Manager() as m:   # no fork of this process
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world,
                 join=True)
        res = dict(out)
    slowest = 10.0 + 5.0 * (world - 1)
    for rank in range(world):
        ms, rate = res[rank]
        assert ms == slowest
        # tokens of all replicas over the slowest replica's time
        assert rate == pytest.approx(world * 8192 * 20 / (slowest / 1e3))


def test_single_process_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_rate(1, 100, 10, 1000.0) == pytest.approx(1000.0)

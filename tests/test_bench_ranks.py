"""bench.py's multi-GPU arithmetic on CPU: two gloo ranks (replicas, no data-path
collective).  The job time is the slowest rank's, and the job's rate counts the work of
every rank over that time."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.0, 5.0][rank]          # rank 1 is the slower replica
        ms = bench.max_over_ranks(local_ms, "cpu")
        out[rank] = (ms, bench.job_rate(100.0, world, ms))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time_and_sum_the_work():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        ms, rate = res[rank]
        assert ms == pytest.approx(5.0)
        assert rate == pytest.approx(2 * 100.0 / 5e-3)


def test_single_rank_keeps_its_own_time():
    assert bench.max_over_ranks(4.0, "cpu") == 4.0
    assert bench.job_rate(10.0, 1, 2.0) == pytest.approx(5000.0)

"""The multi-GPU path is replicas only (independent problems, no exchange step): bench.py's job time is
the slowest rank's and its throughput adds the ranks' work.  Checked with two gloo ranks on the CPU."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [4.0, 6.5][rank]                      # rank 1 is the slow one
        ms = bench.slowest_rank_ms(local, world, torch.device("cpu"))
        out[rank] = (ms, bench.job_throughput(8.796e12, world, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_add_the_work():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, start_method="spawn", join=True)
        res = dict(out)
    assert res[0] == res[1]
    ms, value = res[0]
    assert ms == 6.5
    assert value == pytest.approx(2 * 8.796e12 / 6.5e-3 / 1e12)


def test_single_process_is_its_own_time():
    assert bench.slowest_rank_ms(3.25, 1, torch.device("cpu")) == 3.25
    assert bench.job_throughput(1e12, 1, 1.0) == pytest.approx(1000.0)

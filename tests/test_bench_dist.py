"""The bench's multi-GPU path on CPU: world size 2 over gloo.  Every rank serves
its own batch (independent sequences, no collective on the data path); the job
time is the slowest rank's and the throughput counts every rank's tokens."""
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
        ms = [2.0, 3.5][rank]
        dist.barrier()
        slow = bench.slowest_rank_ms(ms, world)
        out[rank] = (slow, bench.job_throughput(8, world, slow))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    slow, tput = res[0]
    assert slow == 3.5
    assert tput == pytest.approx(2 * 8 / 3.5e-3)


def test_single_rank_needs_no_process_group():
    assert bench.slowest_rank_ms(1.25, 1) == 1.25
    assert bench.job_throughput(8, 1, 2.0) == pytest.approx(4000.0)

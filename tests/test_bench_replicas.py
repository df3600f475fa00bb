"""Host logic of bench.py's multi-replica mode on CPU: world size 2 over gloo.

The path shards by sequence with no data-path collective; the only exchange is
the maximum of the per-rank step times, and the whole-job rate counts the units
of every replica."""
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
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench._dist() == (world, rank)
        mine = [10.0 + 5.0 * rank, 7.0 - rank]          # rank 1 is slower on the first timing only
        got = bench.max_over_ranks(mine, dist)
        out[rank] = got + [bench.whole_job_rate(world, 4096, got[0])]
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_world_size_2():
    world = 2
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        ms_a, ms_b, rate = out[r]
        assert ms_a == 15.0 and ms_b == 7.0            # element-wise max over ranks
        assert rate == pytest.approx(2 * 4096 / 0.015)  # both replicas' units over the slowest time


def test_single_process_passthrough():
    assert bench.max_over_ranks([3.5, 1.25]) == [3.5, 1.25]
    assert bench.whole_job_rate(1, 4096, 50.0) == pytest.approx(81920.0)

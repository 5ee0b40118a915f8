"""The multi-rank host logic of bench.py on CPU: two gloo ranks (no GPU)."""

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
        ms = [12.5, 40.0][rank]  # rank 1 is the slow one
        got = bench.max_over_ranks(ms, world, device="cpu")
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1] == 40.0


def test_weak_throughput_counts_every_rank():
    # 32 rows per rank, 100 steps, 2 ranks, slowest rank took 50 ms
    assert bench.weak_throughput(32, 100, 2, 50.0) == pytest.approx(32 * 100 * 2 / 0.05)
    assert bench.max_over_ranks(3.0, 1) == 3.0

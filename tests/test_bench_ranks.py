"""The multi-rank bench path on CPU: two gloo ranks time different totals;
the slowest rank's time counts and the value covers both ranks' jobs
(weak scaling, no collective on the data path)."""
from __future__ import annotations

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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        total_ms = 100.0 + 20.0 * rank  # rank 1 is the slow one
        ms, value = bench.aggregate_over_ranks(total_ms, steps=10, tokens_per_job=4096, world=world, dist=dist)
        out[rank] = (ms, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    for r in range(world):
        ms, value = out[r]
        assert ms == pytest.approx(12.0)  # max(100, 120) / 10 steps
        assert value == pytest.approx(4096 * 2 / 0.012)


def test_single_rank_needs_no_process_group():
    ms, value = bench.aggregate_over_ranks(50.0, steps=5, tokens_per_job=100, world=1)
    assert ms == 10.0 and value == pytest.approx(100 / 0.010)

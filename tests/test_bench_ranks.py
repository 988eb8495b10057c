"""The multi-rank bench path on CPU.

Batch rows are sharded over the ranks (heads are independent, no exchange):
the ranks' row ranges cover the global batch exactly once, in weak scaling
(B rows per rank) and strong scaling (B rows split).  Two gloo ranks time
different totals: the slowest rank's time counts and the value counts every
token of the global batch once.  `--gpus N` without a process group starts N
ranks under torchrun."""
from __future__ import annotations

import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("scaling", ["weak", "strong"])
@pytest.mark.parametrize("B,world", [(32, 1), (32, 2), (32, 8), (8, 3), (5, 5), (64, 7)])
def test_row_ranges_cover_the_global_batch_once(B, world, scaling):
    rows = [bench.rank_rows(B, world, r, scaling) for r in range(world)]
    Bg = rows[0][2]
    assert all(r[2] == Bg for r in rows)
    assert Bg == (B * world if scaling == "weak" else B)
    covered = [b for b0, nb, _ in rows for b in range(b0, b0 + nb)]
    assert sorted(covered) == list(range(Bg))  # each global row exactly once
    assert all(nb >= 1 for _, nb, _ in rows)
    if scaling == "weak":
        assert all(nb == B for _, nb, _ in rows)
    else:
        assert max(nb for _, nb, _ in rows) - min(nb for _, nb, _ in rows) <= 1


def test_strong_scaling_needs_a_row_per_rank():
    with pytest.raises(ValueError):
        bench.rank_rows(2, 4, 0, "strong")


def _rank(rank, world, port, scaling, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, T = 8, 64
        b0, nb, Bg = bench.rank_rows(B, world, rank, scaling)
        total_ms = 100.0 + 20.0 * rank  # rank 1 is the slow one
        ms, value = bench.aggregate_over_ranks(total_ms, steps=10, tokens_total=Bg * T, world=world, dist=dist)
        gathered = [None] * world
        dist.all_gather_object(gathered, (b0, nb))
        out[rank] = (ms, value, Bg, gathered)
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("scaling", ["weak", "strong"])
def test_two_gloo_ranks_take_the_slowest_time(scaling):
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, _free_port(), scaling, out), nprocs=world, start_method="spawn")
    for r in range(world):
        ms, value, Bg, gathered = out[r]
        assert ms == pytest.approx(12.0)  # max(100, 120) / 10 steps
        assert value == pytest.approx(Bg * 64 / 0.012)  # every global row's tokens, once
        rows = sorted(b for b0, nb in gathered for b in range(b0, b0 + nb))
        assert rows == list(range(Bg))
    assert out[0][2] == (16 if scaling == "weak" else 8)


def test_single_rank_needs_no_process_group():
    ms, value = bench.aggregate_over_ranks(50.0, steps=5, tokens_total=100, world=1)
    assert ms == 10.0 and value == pytest.approx(100 / 0.010)


def test_gpus_flag_starts_torchrun(monkeypatch):
    """`bench.py --gpus 4` outside torchrun re-runs itself as 4 ranks."""
    seen = {}

    def fake_call(cmd):
        seen["cmd"] = cmd
        return 0

    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(bench.subprocess, "call", fake_call)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--gpus", "4", "--steps", "2"])
    with pytest.raises(SystemExit) as e:
        bench.main()
    assert e.value.code == 0
    cmd = seen["cmd"]
    assert cmd[1:3] == ["-m", "torch.distributed.run"] and "--nproc-per-node=4" in cmd
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[-4:] == ["--gpus", "4", "--steps", "2"]


def test_gpus_flag_must_match_world_size(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--gpus", "4"])
    with pytest.raises(SystemExit) as e:
        bench.main()
    assert e.value.code == 2

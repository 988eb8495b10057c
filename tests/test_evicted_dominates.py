"""The inputs of tests/evicted_dominates.py do what they are for (oracle only,
no GPU): the evicted entry holds most of the next query's attention over the
cache it left, at many steps."""
from __future__ import annotations

import synth
from evicted_dominates import build


def test_evicted_entry_dominates_the_next_query():
    w = synth.Workload("evicted_dominates_small", 1, 2, 128, 120, 24, 16, 8, "bf16", 31)
    _, dec, dominated = build(w)
    assert dominated >= 10, dominated  # 11 steps x 2 heads are built
    assert dec[0].shape == (w.T, w.nh, w.d)


def test_evicted_entry_dominates_fp8_and_f32():
    w8 = synth.Workload("evicted_dominates_fp8", 1, 2, 128, 120, 24, 16, 8, "bf16", 32)
    assert build(w8, kv_fp8=True)[2] >= 10
    w32 = synth.Workload("evicted_dominates_f32", 1, 2, 64, 120, 24, 16, 8, "f32", 33)
    assert build(w32)[2] >= 10

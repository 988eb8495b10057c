"""GPU parity of the pipelined decode form where its correction step is
hardest: after many steps the entry just evicted would take most of the next
query's attention (tests/evicted_dominates.py), so the kernel must recompute
that step's partial instead of removing the evicted term.  Every row layout
and storage type: rows resident in shared memory (small caches), streamed
lane-group slabs (long per-CTA chunks), the wide-row layout (grids of two
waves or more), fp32 and fp8 caches.  The cluster form runs the same inputs
as a control."""
from __future__ import annotations

import pytest

import synth
from evicted_dominates import build
from parity_helpers import run_parity

pytestmark = pytest.mark.gpu

W = synth.Workload

CASES = [
    (W("dominated_resident_bf16", 1, 2, 128, 300, 48, 40, 24, "bf16", 41), False),
    (W("dominated_resident_f32_d64", 2, 2, 64, 200, 48, 30, 20, "f32", 42), False),
    (W("dominated_streamed_bf16", 1, 2, 128, 2600, 24, 1300, 1100, "bf16", 43), False),
    (W("dominated_streamed_f32_d64", 1, 2, 64, 2500, 24, 1200, 1200, "f32", 44), False),
    (W("dominated_streamed_fp8", 1, 2, 128, 2600, 24, 1300, 1100, "bf16", 45), True),
    (W("dominated_resident_fp8_d64", 1, 3, 64, 300, 48, 40, 24, "bf16", 46), True),
    (W("dominated_wide_rows", 16, 34, 128, 1100, 12, 501, 500, "bf16", 47), False),
]


@pytest.mark.parametrize("form", ["pipelined", "cluster"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_evicted_entry_dominating_next_query(case, form):
    w, fp8 = case
    prompt, dec, dominated = build(w, kv_fp8=fp8)
    assert dominated >= 8, dominated
    rep, cache = run_parity(w, prompt=prompt, dec=dec, decode_form=form, kv_fp8=fp8)
    print(w.name, form, dominated, rep)
    assert cache.decode_form_used() == form
    assert rep.steps_compared >= w.T

"""Workloads of the exact-tie recipe (synth.tie_prompt / synth.tie_decode).

Dead keys get softmax weight exactly 0, so their scores (and prefill column
sums) stay exactly 0 in fp32 and in fp64: each case below has more dead
heavy-hitter candidates than the selection or the eviction can separate
without the tie rule (prefill keeps the higher of equal positions; eviction
takes the lowest).  Shared by the CPU check that these inputs discriminate
the tie rule and by the GPU parity cases.
"""
from __future__ import annotations

import synth

W = synth.Workload

# (workload, fraction of dead positions)
TIE_CASES = [
    (W("ties_bf16_d128_multitile", 2, 3, 128, 300, 64, 64, 32, "bf16", 9101), 0.8),
    (W("ties_f32_d64", 1, 4, 64, 200, 48, 40, 16, "f32", 9102), 0.9),
    (W("ties_bf16_no_local_block", 1, 2, 128, 100, 40, 24, 0, "bf16", 9103), 0.85),
    (W("ties_bf16_d64_ragged", 2, 2, 64, 333, 40, 50, 40, "bf16", 9104), 0.9),
]
# Budgets of more than 256 slots per cluster CTA (the four-consumer-warp
# cluster kernel) and a prompt long enough for several tensor-core tiles.
TIE_LONG = (W("ties_bf16_long_chunks", 1, 2, 128, 2600, 24, 1300, 1100, "bf16", 9105), 0.6)


def inputs(case):
    w, dead = case
    return synth.tie_prompt(w, dead), synth.tie_decode(w, dead)

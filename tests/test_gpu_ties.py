"""GPU parity at exact ties: the CUDA path's tie rules against the oracle.

The inputs (tests/tie_cases.py, synth.tie_prompt / synth.tie_decode) make
many prefill selections and evictions exact ties in fp32 as well as in fp64:
dead keys get weight exactly 0 and keep score 0.  The harness requires the
GPU's sets to equal the oracle's wherever the oracle's margin is exactly 0
(no resynchronisation there), so these cases pin the kernels' tie rules:
eviction takes the lowest position among equal ranking keys (warp argmin,
cluster decision, last-arriver combine), and the prefill keeps the highest
positions among equal column sums (radix select).  Every decode form, the
fp8 cache and the policy variants run on the same inputs.
"""
from __future__ import annotations

import pytest

from parity_helpers import run_parity
from tie_cases import TIE_CASES, TIE_LONG, inputs

pytestmark = pytest.mark.gpu


def _check(case, **kw):
    w, _ = case
    prompt, dec = inputs(case)
    rep, cache = run_parity(w, prompt=prompt, dec=dec, **kw)
    print(w.name, kw, rep)
    assert rep.ties_prefill > 0 and rep.ties_decode > 0, rep
    assert rep.set_mismatch_prefill == 0 and rep.set_mismatch_decode == 0, rep
    assert rep.steps_compared >= w.T
    return rep, cache


@pytest.mark.parametrize("form", ["per_step", "cooperative", "cluster", "pipelined"])
@pytest.mark.parametrize("case", TIE_CASES, ids=lambda c: c[0].name)
def test_exact_ties_every_form(case, form):
    _, cache = _check(case, decode_form=form)
    assert cache.decode_form_used() == form


@pytest.mark.parametrize("form", ["cooperative", "cluster", "pipelined"])
def test_exact_ties_long_chunks(form):
    _check(TIE_LONG, decode_form=form)


@pytest.mark.parametrize("form", ["per_step", "cluster", "pipelined"])
@pytest.mark.parametrize("case", [TIE_CASES[0], TIE_CASES[2]], ids=lambda c: c[0].name)
def test_exact_ties_fp8_cache(case, form):
    _check(case, decode_form=form, kv_fp8=True)


@pytest.mark.parametrize("policy", [(4, 0), (0, 1), (3, 1)], ids=["sinks", "mean", "sinks_mean"])
@pytest.mark.parametrize("form", ["cooperative", "cluster", "pipelined"])
def test_exact_ties_policies(policy, form):
    _check(TIE_CASES[0], decode_form=form, policy=policy)

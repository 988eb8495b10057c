"""The exact-tie workloads really exercise the tie rule (CPU, oracle only).

On each case the oracle reports selections and evictions with a margin of
exactly 0, and an oracle built with either tie rule reversed (the planted
mistakes "eviction tie goes to the higher position" and "prefill tie keeps
the lower position") reaches a different cache set.  So the GPU parity cases
on these inputs, which require identical sets wherever the margin is 0, fail
for a kernel that breaks ties the other way.
"""
from __future__ import annotations

import os
import tempfile

import numpy as np
import pytest

import oracle
import synth
from test_oracle_pins import MUTANTS
from tie_cases import TIE_CASES, TIE_LONG, inputs


def _run(case, L=None):
    w, _ = case
    (Q, K, V), (q, k, v) = inputs(case)
    cv = lambda x: synth.as_f64(x, w.dtype)
    r = oracle.prefill(cv(Q), cv(K), cv(V), w.k_heavy, w.k_local, _L=L)
    sets0 = [tuple(s) for s in r["state"].sets()]
    st = r["state"]
    o = oracle.decode(st, w.L, cv(q), cv(k), cv(v), w.k_heavy, w.k_local, _L=L)
    return r, sets0, o


def _mutant(name):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "h2o_oracle.c")).read()
    a, b = MUTANTS[name]
    assert src.count(a) == 1
    td = tempfile.mkdtemp()
    path = os.path.join(td, "mut.c")
    open(path, "w").write(src.replace(a, b))
    return oracle.load(oracle.compile_source(path, os.path.join(td, "libmut.so")))


@pytest.mark.parametrize("case", TIE_CASES + [TIE_LONG], ids=lambda c: c[0].name)
def test_tie_cases_have_exact_ties(case):
    r, _, o = _run(case)
    assert np.any(r["margin"] == 0.0), "no exact tie in the prefill selection"
    assert np.sum(o["margin"] == 0.0) >= 5, "too few exact ties among the evictions"


@pytest.mark.parametrize("case", TIE_CASES, ids=lambda c: c[0].name)
def test_reversed_eviction_tie_changes_the_evictions(case):
    _, _, o = _run(case)
    _, _, om = _run(case, _mutant("eviction tie goes to the higher position"))
    assert not np.array_equal(o["evicted"], om["evicted"])


@pytest.mark.parametrize("case", TIE_CASES, ids=lambda c: c[0].name)
def test_reversed_prefill_tie_changes_the_selection(case):
    _, s, _ = _run(case)
    _, sm, _ = _run(case, _mutant("prefill tie keeps the lower position"))
    assert s != sm

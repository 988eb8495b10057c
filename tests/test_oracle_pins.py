"""Pins of the fp64 oracle to things other than itself (CPU only).

* hand-derived worked examples (tests/golden/*.json, exact rationals);
* the Full special case (budget >= sequence length) against a library
  attention routine (torch scaled_dot_product_attention, fp64, CPU);
* the Local special case (k_heavy = 0) against the same routine with a band
  mask, and the closed-form slot set "the k_local most recent positions";
* Definition 4.3 (|S| = k, at most one membership change per step), the
  local block always present, and conservation of score mass
  (live + dropped + evicted = number of attending queries);
* brute force on tiny inputs: enumeration of every heavy-hitter subset for the
  prefill choice, and a history-based replay of the decode loop;
* the policy variants (pinned attention sinks, mean-weight ranking): worked
  examples, the sinks-plus-window case against the library routine with a
  sink+band mask, and a brute-force replay that counts attending queries;
* a planted-mistake check: mutated builds of the oracle source must each fail
  at least one of the pins above.

The method is the H2O summary page's ("H2O: Heavy-Hitter Oracle for Efficient
Generative Inference": "The mechanism", "Algorithm / figure walkthrough",
Definition 4.3).
"""
from __future__ import annotations

import glob
import itertools
import json
import math
import os
import tempfile
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth
from test_oracle_fp8 import FP8_PINS

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GOLDEN_FILES = sorted(glob.glob(os.path.join(GOLDEN, "*.json")))


def _fr(s) -> float:
    return math.inf if s == "inf" else float(Fraction(s))


# --------------------------------------------------------------- golden inputs

def _golden_inputs(g, rng):
    d, L, T = g["d"], g["L"], g["T"]
    if "key" in g:  # identical keys
        key = np.array(g["key"], float)
        K = np.tile(key, (1, L, 1))
        kd = np.tile(key, (T, 1, 1))
        Q = rng.standard_normal((1, L, d))
        qd = rng.standard_normal((T, 1, d))
        V = rng.standard_normal((1, L, d))
        vd = rng.standard_normal((T, 1, d))
    elif "c_prompt" in g:  # designed logits ln(c_j), query 1, value j
        K = np.log(np.array(g["c_prompt"], float)).reshape(1, L, 1)
        kd = np.log(np.array(g["c_decode"], float)).reshape(T, 1, 1)
        Q = np.ones((1, L, 1))
        qd = np.ones((T, 1, 1))
        V = np.arange(L, dtype=float).reshape(1, L, 1)
        vd = np.arange(L, L + T, dtype=float).reshape(T, 1, 1)
    else:  # explicit keys, query 1
        K = np.array(g["keys"], float).reshape(1, L, 1)
        kd = np.array(g.get("decode_keys", []), float).reshape(T, 1, 1)
        Q = np.ones((1, L, 1))
        qd = np.ones((T, 1, 1))
        V = rng.standard_normal((1, L, 1))
        vd = rng.standard_normal((T, 1, 1))
    return Q, K, V, qd, kd, vd


def pin_golden(path, L=None):
    g = json.load(open(path))
    rng = np.random.default_rng(7)
    Q, K, V, qd, kd, vd = _golden_inputs(g, rng)
    kh, kl = g["k_heavy"], g["k_local"]
    pol = dict(n_sink=g.get("n_sink", 0), score_mode=g.get("score_mode", 0))
    r = oracle.prefill(Q, K, V, kh, kl, _L=L, **pol)
    np.testing.assert_allclose(r["colsum"][0], [_fr(x) for x in g["colsum"]], rtol=0, atol=1e-12)
    st = r["state"]
    assert list(st.sets()[0]) == g["prefill_set"]
    if "prefill_set_plain" in g:  # the same prompt under plain summed scores
        plain = oracle.prefill(Q, K, V, kh, kl, _L=L)["state"]
        assert list(plain.sets()[0]) == g["prefill_set_plain"]
    if "evicted_plain" in g:  # the same stream without pinned sinks
        plain = oracle.prefill(Q, K, V, kh, kl, _L=L)["state"]
        assert list(oracle.decode(plain, g["L"], qd, kd, vd, kh, kl, _L=L)["evicted"][:, 0]) == g["evicted_plain"]
    if "prefill_margin" in g:
        assert abs(r["margin"][0] - _fr(g["prefill_margin"])) < 1e-12
    if "prefill_dropped" in g:
        assert abs(r["dropped_mass"][0] - _fr(g["prefill_dropped"])) < 1e-12
    if "lse_exp" in g:
        np.testing.assert_allclose(r["lse"][0], np.log(g["lse_exp"]), rtol=0, atol=1e-12)
    if "O" in g:
        np.testing.assert_allclose(r["O"][0, :, 0], [_fr(x) for x in g["O"]], rtol=0, atol=1e-12)
    if g["T"] == 0:
        return
    o = oracle.decode(st, g["L"], qd, kd, vd, kh, kl, _L=L, **pol)
    assert list(o["evicted"][:, 0]) == g["evicted"]
    np.testing.assert_allclose(o["margin"][:, 0], [_fr(x) for x in g["margin"]], rtol=0, atol=1e-12)
    assert list(st.sets()[0]) == g["final_set"]
    order = np.argsort(st.pos[0][st.pos[0] >= 0])
    np.testing.assert_allclose(st.score[0][st.pos[0] >= 0][order], [_fr(x) for x in g["final_score"]],
                               rtol=0, atol=1e-12)
    assert abs(o["evicted_mass"][0] - _fr(g["evicted_mass"])) < 1e-12
    if "out" in g:
        np.testing.assert_allclose(o["out"][:, 0, 0], [_fr(x) for x in g["out"]], rtol=0, atol=1e-12)
    if "decode_C" in g:  # identical keys: out = mean of V over what the query attends to
        allV = np.concatenate([V[0], vd[:, 0]], 0)
        for t, C in enumerate(g["decode_C"]):
            np.testing.assert_allclose(o["out"][t, 0], allV[C].mean(0), rtol=0, atol=1e-12)


# -------------------------------------------------------- library special cases

def _sdpa(q, k, v, mask):
    """torch's attention routine in fp64 on CPU: q [n, d], k/v [m, d], mask [n, m] bool."""
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None, None], torch.from_numpy(k)[None, None], torch.from_numpy(v)[None, None],
        attn_mask=torch.from_numpy(mask)[None, None]).numpy()[0, 0]


def _rand(nh, L, T, d, seed):
    rng = np.random.default_rng(seed)
    f = lambda *s: rng.standard_normal(s)
    return f(nh, L, d), f(nh, L, d) * 1.5, f(nh, L, d), f(T, nh, d), f(T, nh, d) * 1.5, f(T, nh, d)


def pin_full_equals_library(L=None):
    """Budget >= L+T: nothing is ever evicted, so H2O is exact causal attention
    over the whole stream, and each final score is a causal-softmax column sum."""
    nh, Lp, T, d = 3, 7, 9, 8
    Q, K, V, qd, kd, vd = _rand(nh, Lp, T, d, 11)
    r = oracle.prefill(Q, K, V, 10, 6, _L=L)
    o = oracle.decode(r["state"], Lp, qd, kd, vd, 10, 6, _L=L)
    assert (o["evicted"] == -1).all()
    n = Lp + T
    causal = np.tril(np.ones((n, n), bool))
    for h in range(nh):
        q = np.concatenate([Q[h], qd[:, h]]); k = np.concatenate([K[h], kd[:, h]])
        v = np.concatenate([V[h], vd[:, h]])
        ref = _sdpa(q, k, v, causal)
        np.testing.assert_allclose(r["O"][h], ref[:Lp], rtol=0, atol=1e-12)
        np.testing.assert_allclose(o["out"][:, h], ref[Lp:], rtol=0, atol=1e-12)
        logits = torch.from_numpy(q @ k.T / math.sqrt(d)).masked_fill(~torch.from_numpy(causal), -math.inf)
        np.testing.assert_allclose(r["lse"][h], torch.logsumexp(logits[:Lp, :Lp], 1).numpy(), rtol=0, atol=1e-12)
        P = torch.softmax(logits, 1).numpy()
        np.testing.assert_allclose(r["colsum"][h], P[:Lp, :Lp].sum(0), rtol=0, atol=1e-12)
        st = r["state"]
        live = st.pos[h] >= 0
        np.testing.assert_allclose(st.score[h][live][np.argsort(st.pos[h][live])], P.sum(0), rtol=0,
                                   atol=1e-12)


def pin_local_equals_library(L=None):
    """k_heavy = 0: the eviction candidates are exactly the oldest entry, so the
    cache is a sliding window of the k_local newest positions and each decode
    query attends to positions p-k_local .. p."""
    nh, Lp, T, d, kl = 2, 10, 12, 8, 4
    Q, K, V, qd, kd, vd = _rand(nh, Lp, T, d, 12)
    r = oracle.prefill(Q, K, V, 0, kl, _L=L)
    st = r["state"]
    for h in range(nh):
        assert list(st.sets()[h]) == list(range(Lp - kl, Lp))
    o = oracle.decode(st, Lp, qd, kd, vd, 0, kl, _L=L)
    for t in range(T):
        p = Lp + t
        assert (o["evicted"][t] == p - kl).all()
    for h in range(nh):
        assert list(st.sets()[h]) == list(range(Lp + T - kl, Lp + T))
        q = np.concatenate([Q[h], qd[:, h]]); k = np.concatenate([K[h], kd[:, h]])
        v = np.concatenate([V[h], vd[:, h]])
        n = Lp + T
        i, j = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
        band = (j <= i) & ((i < Lp) | (j >= i - kl))
        ref = _sdpa(q, k, v, band)
        np.testing.assert_allclose(o["out"][:, h], ref[Lp:], rtol=0, atol=1e-12)


# --------------------------------------------------------------- invariants

def pin_def43_and_mass(L=None):
    """Definition 4.3 (|S| = k, at most one change per step), the newest
    k_local positions always cached, and score mass conservation."""
    for (nh, Lp, T, d, kh, kl) in [(3, 40, 60, 16, 5, 7), (2, 6, 30, 8, 4, 3), (2, 20, 25, 8, 6, 0)]:
        Q, K, V, qd, kd, vd = _rand(nh, Lp, T, d, 13 + Lp)
        k = kh + kl
        r = oracle.prefill(Q, K, V, kh, kl, _L=L)
        st = r["state"]
        total_dropped = r["dropped_mass"].copy()
        prev = st.sets()
        for t in range(T):
            p = Lp + t
            o = oracle.decode(st, p, qd[t:t + 1], kd[t:t + 1], vd[t:t + 1], kh, kl, _L=L)
            total_dropped += o["evicted_mass"]
            cur = st.sets()
            for h in range(nh):
                c, pr = set(cur[h].tolist()), set(prev[h].tolist())
                assert len(c) == min(k, Lp + t + 1)
                assert len(c - pr) <= 1 and len(pr - c) <= 1
                ev = o["evicted"][0, h]
                if ev == -1:
                    assert c == pr | {p}
                elif ev == p:
                    assert c == pr
                else:
                    assert c == (pr - {ev}) | {p} and ev <= p - kl
                assert set(range(max(0, p - kl + 1), p + 1)) <= c
                live = st.score[h][st.pos[h] >= 0].sum()
                assert abs(live + total_dropped[h] - (Lp + t + 1)) < 1e-9 * (Lp + t + 1)
            prev = cur


# --------------------------------------------------------------- brute force

def pin_select_bruteforce(L=None):
    """The prefill heavy set is the subset of size k_heavy with the largest
    total column-sum mass (enumerated over every subset)."""
    for seed in range(4):
        Q, K, V, *_ = _rand(1, 12, 0, 6, 100 + seed)
        kh, kl = 3, 3
        r = oracle.prefill(Q, K, V, kh, kl, _L=L)
        cs = r["colsum"][0]
        nc = 12 - kl
        best = max(itertools.combinations(range(nc), kh), key=lambda s: sum(cs[j] for j in s))
        got = [j for j in r["state"].sets()[0] if j < nc]
        assert sorted(best) == got
        assert abs(sum(cs) - 12) < 1e-12  # every query's weights sum to one


def pin_decode_bruteforce(L=None):
    """Replay of the decode loop from the full weight history: each score is
    re-summed from every weight the position ever received (prompt column sum
    included), and the evicted entry is found by comparing every candidate with
    every other."""
    nh, Lp, T, d, kh, kl = 2, 6, 14, 4, 2, 2
    Q, K, V, qd, kd, vd = _rand(nh, Lp, T, d, 21)
    r = oracle.prefill(Q, K, V, kh, kl, _L=L)
    st = r["state"]
    o = oracle.decode(st, Lp, qd, kd, vd, kh, kl, _L=L)
    for h in range(nh):
        keys = {j: K[h, j] for j in range(Lp)}
        vals = {j: V[h, j] for j in range(Lp)}
        history = {j: [r["colsum"][h, j]] for j in range(Lp)}
        # rebuild S_0 from the prompt scores by enumeration (largest mass subset)
        nc = Lp - kl
        heavy = max(itertools.combinations(range(nc), kh), key=lambda s: sum(history[j][0] for j in s))
        S = set(heavy) | set(range(Lp - kl, Lp))
        for t in range(T):
            p = Lp + t
            keys[p], vals[p] = kd[t, h], vd[t, h]
            C = sorted(S | {p})
            logits = [float(np.dot(qd[t, h], keys[j])) / math.sqrt(d) for j in C]
            mx = max(logits)
            ex = [math.exp(x - mx) for x in logits]
            z = sum(ex)
            out = sum((e / z) * vals[j] for e, j in zip(ex, C))
            np.testing.assert_allclose(o["out"][t, h], out, rtol=0, atol=1e-12)
            for e, j in zip(ex, C):
                history.setdefault(j, []).append(e / z)
            if len(C) <= kh + kl:
                assert o["evicted"][t, h] == -1
                S = set(C)
                continue
            E = [j for j in C if j <= p - kl]
            F = {j: math.fsum(history[j]) for j in E}
            loser = [j for j in E if all((F[j], j) <= (F[i], i) for i in E)]
            assert len(loser) == 1
            assert o["evicted"][t, h] == loser[0]
            S = set(C) - {loser[0]}
        assert set(st.sets()[h].tolist()) == S
        live = st.pos[h] >= 0
        for pos, sc in zip(st.pos[h][live], st.score[h][live]):
            assert abs(sc - math.fsum(history[int(pos)])) < 1e-12


# ------------------------------------------------------- policy variants

def pin_streaming_equals_library(L=None):
    """n_sink = k_heavy: every heavy slot is a pinned sink, so the cache is the
    first n_sink positions plus a window of the k_local newest, each decode
    query at p attends to j < n_sink and p-k_local <= j <= p, and the entry
    evicted at p is p-k_local."""
    nh, Lp, T, d, ns, kl = 2, 12, 15, 8, 3, 4
    Q, K, V, qd, kd, vd = _rand(nh, Lp, T, d, 31)
    r = oracle.prefill(Q, K, V, ns, kl, _L=L, n_sink=ns)
    st = r["state"]
    for h in range(nh):
        assert list(st.sets()[h]) == list(range(ns)) + list(range(Lp - kl, Lp))
    o = oracle.decode(st, Lp, qd, kd, vd, ns, kl, _L=L, n_sink=ns)
    for t in range(T):
        assert (o["evicted"][t] == Lp + t - kl).all()
    for h in range(nh):
        assert list(st.sets()[h]) == list(range(ns)) + list(range(Lp + T - kl, Lp + T))
        q = np.concatenate([Q[h], qd[:, h]]); k = np.concatenate([K[h], kd[:, h]])
        v = np.concatenate([V[h], vd[:, h]])
        n = Lp + T
        i, j = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
        mask = (j <= i) & ((i < Lp) | (j < ns) | (j >= i - kl))
        np.testing.assert_allclose(o["out"][:, h], _sdpa(q, k, v, mask)[Lp:], rtol=0, atol=1e-12)


def pin_policy_bruteforce(L=None):
    """Replay of the loop for the variants from the full weight history: the
    number of queries that attended to each position is counted, not derived;
    the prefill heavy set is found by enumerating subsets of the non-sink
    candidates; the evicted entry by comparing every candidate with every
    other."""
    nh, Lp, T, d, kh, kl = 2, 9, 14, 4, 3, 2
    Q, K, V, qd, kd, vd = _rand(nh, Lp, T, d, 41)
    for ns, mode in [(1, 0), (0, 1), (2, 1), (3, 1)]:
        r = oracle.prefill(Q, K, V, kh, kl, _L=L, n_sink=ns, score_mode=mode)
        st = r["state"]
        o = oracle.decode(st, Lp, qd, kd, vd, kh, kl, _L=L, n_sink=ns, score_mode=mode)
        causal = np.tril(np.ones((Lp, Lp), bool))
        for h in range(nh):
            keys = {j: K[h, j] for j in range(Lp)}
            history = {j: [r["colsum"][h, j]] for j in range(Lp)}
            seen = {j: int(causal[:, j].sum()) for j in range(Lp)}  # prompt queries that attended to j

            def rank(j):
                return math.fsum(history[j]) / seen[j] if mode else math.fsum(history[j])

            nc = Lp - kl
            free = [j for j in range(nc) if j >= ns]
            heavy = max(itertools.combinations(free, kh - ns),
                        key=lambda s: (sum(rank(j) for j in s), sorted(s, reverse=True)))
            S = set(range(ns)) | set(heavy) | set(range(Lp - kl, Lp))
            assert set(r["state"].sets()[h].tolist()) >= set(range(ns))
            for t in range(T):
                p = Lp + t
                keys[p] = kd[t, h]
                C = sorted(S | {p})
                logits = [float(np.dot(qd[t, h], keys[j])) / math.sqrt(d) for j in C]
                mx = max(logits)
                ex = [math.exp(x - mx) for x in logits]
                z = sum(ex)
                for e, j in zip(ex, C):
                    history.setdefault(j, []).append(e / z)
                    seen[j] = seen.get(j, 0) + 1
                if len(C) <= kh + kl:
                    assert o["evicted"][t, h] == -1
                    S = set(C)
                    continue
                E = [j for j in C if ns <= j <= p - kl]
                loser = [j for j in E if all((rank(j), j) <= (rank(i), i) for i in E)]
                assert len(loser) == 1
                assert o["evicted"][t, h] == loser[0], (ns, mode, t, h)
                S = set(C) - {loser[0]}
            assert set(st.sets()[h].tolist()) == S
            live = st.pos[h] >= 0
            for pos, sc in zip(st.pos[h][live], st.score[h][live]):
                assert abs(sc - math.fsum(history[int(pos)])) < 1e-12


def pin_policy_invariants(L=None):
    """Definition 4.3 and score-mass conservation hold for the variants too,
    and the first n_sink positions never leave the cache."""
    nh, Lp, T, d, kh, kl = 3, 30, 50, 8, 6, 5
    Q, K, V, qd, kd, vd = _rand(nh, Lp, T, d, 51)
    for ns, mode in [(2, 0), (0, 1), (4, 1)]:
        r = oracle.prefill(Q, K, V, kh, kl, _L=L, n_sink=ns, score_mode=mode)
        st = r["state"]
        total = r["dropped_mass"].copy()
        prev = st.sets()
        for t in range(T):
            p = Lp + t
            o = oracle.decode(st, p, qd[t:t + 1], kd[t:t + 1], vd[t:t + 1], kh, kl, _L=L, n_sink=ns,
                              score_mode=mode)
            total += o["evicted_mass"]
            cur = st.sets()
            for h in range(nh):
                c, pr = set(cur[h].tolist()), set(prev[h].tolist())
                assert len(c) == kh + kl and len(c - pr) <= 1 and len(pr - c) <= 1
                assert set(range(ns)) <= c and set(range(p - kl + 1, p + 1)) <= c
                live = st.score[h][st.pos[h] >= 0].sum()
                assert abs(live + total[h] - (p + 1)) < 1e-9 * (p + 1)
            prev = cur


def test_policy_arguments_checked():
    Q, K, V, *_ = _rand(1, 8, 0, 4, 3)
    with pytest.raises(ValueError):
        oracle.prefill(Q, K, V, 2, 2, n_sink=3)
    with pytest.raises(ValueError):
        oracle.prefill(Q, K, V, 2, 2, score_mode=2)


PINS = [pin_full_equals_library, pin_local_equals_library, pin_def43_and_mass, pin_select_bruteforce,
        pin_decode_bruteforce, pin_streaming_equals_library, pin_policy_bruteforce,
        pin_policy_invariants] + FP8_PINS + [
    (lambda path: (lambda L=None: pin_golden(path, L)))(p) for p in GOLDEN_FILES]


# ------------------------------------------------------------------- tests

@pytest.mark.parametrize("path", GOLDEN_FILES, ids=lambda p: os.path.basename(p))
def test_golden(path):
    pin_golden(path)


def test_golden_files_present():
    assert len(GOLDEN_FILES) >= 5


def test_full_equals_library():
    pin_full_equals_library()


def test_local_equals_library():
    pin_local_equals_library()


def test_def43_and_mass():
    pin_def43_and_mass()


def test_select_bruteforce():
    pin_select_bruteforce()


def test_decode_bruteforce():
    pin_decode_bruteforce()


def test_streaming_equals_library():
    pin_streaming_equals_library()


def test_policy_bruteforce():
    pin_policy_bruteforce()


def test_policy_invariants():
    pin_policy_invariants()


def test_naive_topk_is_not_h2o():
    """The page warns that a fresh Top-K each step is a different algorithm:
    keeping the k entries with the largest weight of the current step alone
    gives other cache sets than H2O on the tiny workload."""
    w = synth.TINY
    Q, K, V = (synth.as_f64(x, w.dtype) for x in synth.prompt(w))
    qd, kd, vd = (synth.as_f64(x, w.dtype) for x in synth.decode(w, 0, w.T))
    r = oracle.prefill(Q, K, V, w.k_heavy, w.k_local)
    st = r["state"]
    o = oracle.decode(st, w.L, qd, kd, vd, w.k_heavy, w.k_local)
    h2o_sets = st.sets()
    differs = False
    for h in range(w.nh):
        naive = set(np.argsort(-r["colsum"][h])[:w.k].tolist())
        allK = np.concatenate([K[h], kd[:, h]])
        for t in range(w.T):
            p = w.L + t
            C = sorted(naive | {p})
            lg = allK[C] @ qd[t, h] / math.sqrt(w.d)
            keep = np.argsort(-lg, kind="stable")[:w.k]
            naive = {C[i] for i in keep}
        differs |= naive != set(h2o_sets[h].tolist())
    assert differs


MUTANTS = {
    "query does not attend to itself": ("w[n] = scale * dot(qt, kt, d);", "w[n] = -INFINITY;"),
    "eviction tie goes to the higher position": ("(sj == best_s && pj < best_p)", "(sj == best_s && pj > best_p)"),
    "local block one position too small": ("if (pj > p - kl) continue;", "if (pj >= p - kl) continue;"),
    "column sum indexed by the query": ("for (int j = 0; j <= i; ++j) F[j] += e[j] / l;",
                                        "for (int j = 0; j <= i; ++j) F[i] += e[j] / l;"),
    "new entry starts at score 0": ("score[best] = w_new;", "score[best] = 0.0;"),
    "softmax scale dropped": ("const double scale = 1.0 / sqrt((double)d);\n  double *w", "const double scale = 1.0;\n  double *w"),
    "prefill tie keeps the lower position": ("return (a->j > b->j) ? -1 : (a->j < b->j) ? 1 : 0;",
                                             "return (a->j < b->j) ? -1 : (a->j > b->j) ? 1 : 0;"),
    "evicted mass not recorded": ("if (evicted_mass) *evicted_mass += score[best];", ";"),
    "new value left out of the output": ("for (int c = 0; c < d; ++c) o[c] += w[n] * vt[c];", ";"),
    "base-2 log-sum-exp": ("if (lse) lse[i] = m + log(l);", "if (lse) lse[i] = m + log2(l);"),
    "heavy candidates include the local block": ("const int nc = L - kl;", "const int nc = L;"),
    "scores not accumulated": ("for (int j = 0; j < n; ++j) score[j] += w[j];", ";"),
    "sinks not protected in decode": ("if (pj < ns) continue;", ";"),
    "sinks not kept by the prefill": ("for (int j = 0; j < ns; ++j) keep[n++] = j;", ";"),
    "decode age counts one query too few": ("p - pj + 1, mode)", "p - pj, mode)"),
    "prefill age counts one query too many": ("rank_key(F[j], L - j, mode)", "rank_key(F[j], L - j + 1, mode)"),
    "decode ignores the mean ranking": ("p - pj + 1, mode)", "p - pj + 1, 0)"),
    "prefill ignores the mean ranking": ("rank_key(F[j], L - j, mode)", "rank_key(F[j], L - j, 0)"),
    "fp8 rows not scaled back": ("e4m3_round((double)((float)x[c] / sc)) * (double)sc : 0.0",
                                 "e4m3_round((double)((float)x[c] / sc)) : 0.0"),
    "fp8 rounding ties away from zero": ("nearbyint(a / quantum)", "round(a / quantum)"),
    "fp8 subnormal step too fine": ("double quantum = ldexp(1.0, -9);", "double quantum = ldexp(1.0, -10);"),
    "fp8 scale for a 240 maximum": ("amax / 448.0f", "amax / 240.0f"),
    "fp8 decode rows stored unquantised": ("store_row(kt, d, fp8, Ks + (size_t)best * d",
                                           "store_row(kt, d, 0, Ks + (size_t)best * d"),
    "fp8 prefill rows stored unquantised": ("store_row(K + (size_t)j * d, d, fp8,", "store_row(K + (size_t)j * d, d, 0,"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    """Each planted mistake in the oracle's source must make a pin fail."""
    src = open(os.path.join(os.path.dirname(oracle.__file__), "h2o_oracle.c")).read()
    a, b = MUTANTS[name]
    assert src.count(a) == 1, f"mutation anchor not found: {a!r}"
    with tempfile.TemporaryDirectory() as td:
        path = os.path.join(td, "mut.c")
        open(path, "w").write(src.replace(a, b))
        L = oracle.load(oracle.compile_source(path, os.path.join(td, "libmut.so")))
        failed = []
        for pin in PINS:
            try:
                pin(L)
            except (AssertionError, ValueError):
                failed.append(pin)
        assert failed, f"no pin caught: {name}"

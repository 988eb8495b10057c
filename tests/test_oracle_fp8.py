"""Pins of the oracle's fp8 cache rows (kv_fp8), CPU only.

The cache stores each K/V row as e4m3 codes with one fp32 scale per row
(scale = amax / 448, code = nearest-even e4m3 of x / scale) — the
quantisation that the explainer page's "Limitations" section says H2O
composes with.  Pinned against torch's own float8_e4m3fn conversion (a
library rounding routine), against the format's error bound, and by a
brute-force replay of the decode loop whose cached rows are quantised with
torch.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import synth


def torch_fp8_row(x: np.ndarray):
    """Row as an fp8 cache holds it, computed with torch: fp32 scale, fp32
    division, torch's e4m3 conversion; returns (values, scale)."""
    xf = torch.from_numpy(x.astype(np.float32))
    amax = xf.abs().max()
    scale = amax / torch.tensor(448.0, dtype=torch.float32)
    if float(scale) == 0.0:
        return np.zeros_like(x), 0.0
    codes = (xf / scale).to(torch.float8_e4m3fn).to(torch.float64)
    return (codes * float(scale)).numpy(), float(scale)


def _bf16_grid():
    """Every positive bf16 value in [2^-12, 448], both signs: they cover all
    e4m3 binades, the subnormal range and the exact midpoints."""
    bits = np.arange(0x3980, 0x43E1, dtype=np.uint32)  # 2^-12 .. 448 as bf16 patterns
    v = (bits << 16).view(np.float32).astype(np.float64)
    v = v[(v >= 2.0 ** -12) & (v <= 448.0)]
    return np.concatenate([v, -v])


def _prefill_rows(rows: np.ndarray, d: int, lib=None):
    """Prefill whose every row is kept (L <= k) so the state holds each K row
    as the fp8 cache stores it."""
    L = rows.shape[0]
    K = rows.reshape(1, L, d)
    Q = np.zeros_like(K)
    r = oracle.prefill(Q, K, K, L, 0, _L=lib, kv_fp8=True)
    st = r["state"]
    order = np.argsort(st.pos[0])
    return st.K[0][order], st.Ksc[0][order]


def pin_fp8_rounding(L=None):
    """Every bf16 value in [2^-12, 448] of either sign, stored with scale 1,
    reads back as torch's e4m3 conversion of it."""
    d = 64
    grid = _bf16_grid()
    per = d - 1
    n = -(-grid.size // per)
    vals = np.concatenate([grid, np.ones(n * per - grid.size)])
    rows = np.concatenate([np.full((n, 1), 448.0), vals.reshape(n, per)], 1)  # amax 448 -> scale 1
    got, sc = _prefill_rows(rows, d, L)
    assert (sc == 1.0).all()
    for i in range(n):
        want, s = torch_fp8_row(rows[i])
        assert s == 1.0
        np.testing.assert_array_equal(got[i], want)


def pin_fp8_rows(L=None):
    """Rows of any magnitude: values and scales equal torch's, within the
    format's error bound; an all-zero row stores scale 0."""
    rng = np.random.default_rng(3)
    d = 128
    rows = synth.as_f64(synth.f32_to_bf16_bits((rng.standard_normal((40, d)) *
                                                 np.exp(rng.uniform(-8, 8, (40, 1)))).astype(np.float32)), "bf16")
    rows[5] = 0.0  # an all-zero row stores scale 0
    got, sc = _prefill_rows(rows, d, L)
    for i in range(rows.shape[0]):
        want, s = torch_fp8_row(rows[i])
        np.testing.assert_array_equal(got[i], want)
        assert sc[i] == s
        # e4m3 keeps 3 mantissa bits: error <= half a quantum, 2^-4 relative
        # for normal codes and 2^-10 * scale in the subnormal range
        bound = np.maximum(np.abs(rows[i]) * 2.0 ** -4, 2.0 ** -10 * s)
        assert (np.abs(got[i] - rows[i]) <= bound * (1 + 1e-6)).all()
    assert sc[5] == 0.0 and (got[5] == 0).all()


def _rand(nh, L, T, d, seed):
    rng = np.random.default_rng(seed)
    f = lambda *s: synth.as_f64(synth.f32_to_bf16_bits(rng.standard_normal(s).astype(np.float32)), "bf16")
    return f(nh, L, d), f(nh, L, d), f(nh, L, d), f(T, nh, d), f(T, nh, d), f(T, nh, d)


def pin_fp8_replay(L=None):
    """Replay with torch-quantised cache rows: the prompt is attended at input
    precision, kept rows are stored as fp8, each decode query attends the
    stored rows plus its own token at input precision, and the new row is
    stored as fp8 after the eviction."""
    nh, Lp, T, d, kh, kl = 2, 10, 16, 8, 3, 3
    Q, K, V, qd, kd, vd = _rand(nh, Lp, T, d, 61)
    r = oracle.prefill(Q, K, V, kh, kl, _L=L, kv_fp8=True)
    plain = oracle.prefill(Q, K, V, kh, kl, _L=L)
    np.testing.assert_array_equal(r["colsum"], plain["colsum"])  # the prompt itself is not quantised
    np.testing.assert_array_equal(r["O"], plain["O"])
    st = r["state"]
    o = oracle.decode(st, Lp, qd, kd, vd, kh, kl, _L=L, kv_fp8=True)
    for h in range(nh):
        S = {}
        keep = plain["state"].sets()[h]
        for p in keep:
            S[int(p)] = [torch_fp8_row(K[h, p])[0], torch_fp8_row(V[h, p])[0], r["colsum"][h, p]]
        for t in range(T):
            p = Lp + t
            C = sorted(S) + [p]
            keys = [S[j][0] for j in C[:-1]] + [kd[t, h]]
            vals = [S[j][1] for j in C[:-1]] + [vd[t, h]]
            lg = [float(np.dot(qd[t, h], kk)) / math.sqrt(d) for kk in keys]
            mx = max(lg)
            ex = [math.exp(x - mx) for x in lg]
            z = sum(ex)
            out = sum((e / z) * v for e, v in zip(ex, vals))
            np.testing.assert_allclose(o["out"][t, h], out, rtol=0, atol=1e-12)
            for e, j in zip(ex[:-1], C[:-1]):
                S[j][2] += e / z
            new = [torch_fp8_row(kd[t, h])[0], torch_fp8_row(vd[t, h])[0], ex[-1] / z]
            if len(C) <= kh + kl:
                assert o["evicted"][t, h] == -1
                S[p] = new
                continue
            E = [j for j in C if j <= p - kl]
            sc = {j: (S[j][2] if j != p else new[2]) for j in E}
            loser = min(E, key=lambda j: (sc[j], j))
            assert o["evicted"][t, h] == loser
            if loser != p:
                del S[loser]
                S[p] = new
        live = st.pos[h] >= 0
        for pos, kk, vv, sc in zip(st.pos[h][live], st.K[h][live], st.V[h][live], st.score[h][live]):
            np.testing.assert_array_equal(kk, S[int(pos)][0])
            np.testing.assert_array_equal(vv, S[int(pos)][1])
            assert abs(sc - S[int(pos)][2]) < 1e-12


def test_rounding_matches_torch_on_every_bf16_value():
    pin_fp8_rounding()


def test_rows_match_torch_and_error_bound():
    pin_fp8_rows()


def test_fp8_replay():
    pin_fp8_replay()


FP8_PINS = [pin_fp8_rounding, pin_fp8_rows, pin_fp8_replay]


def test_fp8_scales_exported_and_differs_from_bf16():
    """The fp8 cache changes the decode outputs (by up to the quantisation
    error) and records one scale per stored row."""
    Q, K, V, qd, kd, vd = _rand(2, 12, 6, 16, 62)
    a = oracle.prefill(Q, K, V, 4, 4, kv_fp8=True)
    b = oracle.prefill(Q, K, V, 4, 4)
    oa = oracle.decode(a["state"], 12, qd, kd, vd, 4, 4, kv_fp8=True)
    ob = oracle.decode(b["state"], 12, qd, kd, vd, 4, 4)
    assert np.abs(oa["out"] - ob["out"]).max() > 0
    assert np.abs(oa["out"] - ob["out"]).max() < 0.2
    st = a["state"]
    for h in range(2):
        for s in range(8):
            want = np.abs(st.K[h, s]).max() / 448.0
            assert abs(st.Ksc[h, s] - want) <= 1e-6 * want
    assert (b["state"].Ksc == 1.0).all()


def test_fp8_flag_checked():
    Q, K, V, *_ = _rand(1, 8, 0, 4, 3)
    with pytest.raises(ValueError):
        oracle.prefill(Q, K, V, 2, 2, kv_fp8=2)

"""Seeded synthetic inputs for the H2O decode/prefill path.

This module is shared by the CUDA path's callers (tests, bench) and by the
oracle's callers.  It draws random numbers and rounds them to the storage
dtype; it holds none of the method's arithmetic (no attention, no scores, no
eviction).

Recipe, per (batch b, head h) — the workload family of the H2O paper's
OPT-6.7B / OPT-30B serving experiments ("Results and evidence", throughput at a
20% heavy-hitter budget), shaped synthetically because the models and task
data are not available:

* ``u``: a unit direction, ``z / ||z||`` with ``z ~ N(0, I_d)``;
* keys ``K_j = N(0, I_d) + s_j * u`` with ``s_j ~ Pareto(alpha=1.5)``
  (Type I, scale 1: ``s = (1-U)^(-1/1.5)``) clipped to 8, so a few keys
  carry a large component along ``u`` (power-law heavy hitters);
* queries ``q = N(0, I_d) + 2u``;
* values ``V ~ N(0, 1)``;
* optionally a planted fraction of positions (over prompt and decode) gets
  ``s_j = 8`` exactly.

Every (b, h) has its own counter-addressed stream (``numpy`` SeedSequence keyed
by ``[seed, b, h, segment]``), so any head, and any chunk of decode steps, can
be regenerated on its own.  Values are produced in fp32 and, for bf16 runs,
rounded once to bf16 with round-to-nearest-even; every consumer sees the same
bits.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

BASE_SEED = 20230624
DECODE_CHUNK = 256  # decode steps per generator segment
PARETO_ALPHA = 1.5
PARETO_CLIP = 8.0
QUERY_SHIFT = 2.0


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape of one H2O run: B x H heads of width d, prompt length L,
    T decode steps, budget k = k_heavy + k_local, storage dtype."""

    name: str
    B: int
    H: int
    d: int
    L: int
    T: int
    k_heavy: int
    k_local: int
    dtype: str  # "f32" or "bf16"
    seed: int
    planted_frac: float = 0.0

    @property
    def k(self) -> int:
        return self.k_heavy + self.k_local

    @property
    def nh(self) -> int:
        return self.B * self.H

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads: a tiny fp32 correctness case, then single layers shaped
# like OPT-6.7B and OPT-30B at a 20% KV budget, a prefill-heavy serving case
# with planted hitters, and a long stream with an H2O-256 budget.
CONFIGS = [
    Workload("tiny_f32_B1H2d64_L64_T64_k16+16", 1, 2, 64, 64, 64, 16, 16, "f32", BASE_SEED + 0),
    Workload("opt6.7b_B8H32d128_L2048_T512_k256+256", 8, 32, 128, 2048, 512, 256, 256, "bf16", BASE_SEED + 1),
    Workload("opt30b_B64H56d128_L1024_T1024_k204+204", 64, 56, 128, 1024, 1024, 204, 204, "bf16", BASE_SEED + 2),
    Workload("prefill_heavy_B32H32d128_L8192_T256_k845+845", 32, 32, 128, 8192, 256, 845, 845, "bf16",
             BASE_SEED + 3, planted_frac=0.05),
    Workload("long_stream_B1H32d128_L256_T4194304_k128+128", 1, 32, 128, 256, 4194304, 128, 128, "bf16",
             BASE_SEED + 4),
]
TINY, OPT_6_7B, OPT_30B, PREFILL_HEAVY, LONG_STREAM = CONFIGS


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(w: Workload, b: int, h: int, segment: int) -> np.random.Generator:
    return np.random.default_rng([w.seed, b, h, segment])


def _direction(w: Workload, b: int, h: int) -> np.ndarray:
    z = _rng(w, b, h, 0).standard_normal(w.d)
    return (z / np.linalg.norm(z)).astype(np.float32)


def _planted(w: Workload, b: int, h: int) -> np.ndarray:
    """Sorted positions (over prompt + decode) whose s_j is pinned to the clip."""
    if w.planted_frac <= 0.0:
        return np.zeros(0, dtype=np.int64)
    n_pos = w.L + w.T
    count = int(round(w.planted_frac * n_pos))
    return np.sort(_rng(w, b, h, 1).choice(n_pos, size=count, replace=False))


def _draw_rows(rng: np.random.Generator, n: int, d: int, u: np.ndarray,
               first_pos: int, planted: np.ndarray):
    """n consecutive positions: returns fp32 (q, k, v), each [n, d]."""
    kn = rng.standard_normal((n, d), dtype=np.float32)
    uni = rng.random(n)
    s = np.minimum((1.0 - uni) ** (-1.0 / PARETO_ALPHA), PARETO_CLIP)
    if planted.size:
        sel = planted[(planted >= first_pos) & (planted < first_pos + n)] - first_pos
        s[sel] = PARETO_CLIP
    qn = rng.standard_normal((n, d), dtype=np.float32)
    v = rng.standard_normal((n, d), dtype=np.float32)
    k = kn + s.astype(np.float32)[:, None] * u[None, :]
    q = qn + np.float32(QUERY_SHIFT) * u[None, :]
    return q, k, v


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(x) if dtype == "bf16" else np.ascontiguousarray(x, dtype=np.float32)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _heads(w: Workload, heads):
    return list(range(w.nh)) if heads is None else [int(x) for x in heads]


def prompt(w: Workload, heads=None):
    """Prompt Q, K, V of the selected heads (flat index b*H + h), each
    [n_heads, L, d] in storage form (fp32, or uint16 bf16 bits)."""
    hs = _heads(w, heads)
    st = np.uint16 if w.dtype == "bf16" else np.float32
    Q = np.empty((len(hs), w.L, w.d), st)
    K = np.empty_like(Q)
    V = np.empty_like(Q)

    def one(i):
        b, h = divmod(hs[i], w.H)
        u = _direction(w, b, h)
        q, k, v = _draw_rows(_rng(w, b, h, 2), w.L, w.d, u, 0, _planted(w, b, h))
        Q[i], K[i], V[i] = _store(q, w.dtype), _store(k, w.dtype), _store(v, w.dtype)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(len(hs))))
    return Q, K, V


def decode(w: Workload, t0: int, n: int, heads=None):
    """Decode-step inputs q_t, k_t, v_t for steps t0 .. t0+n-1 of the selected
    heads, each [n, n_heads, d] (step-major) in storage form."""
    hs = _heads(w, heads)
    st = np.uint16 if w.dtype == "bf16" else np.float32
    q = np.empty((n, len(hs), w.d), st)
    k = np.empty_like(q)
    v = np.empty_like(q)
    c_lo, c_hi = t0 // DECODE_CHUNK, (t0 + n - 1) // DECODE_CHUNK if n > 0 else -1

    def one(i):
        b, h = divmod(hs[i], w.H)
        u = _direction(w, b, h)
        pl = _planted(w, b, h)
        for c in range(c_lo, c_hi + 1):
            cs = c * DECODE_CHUNK
            qq, kk, vv = _draw_rows(_rng(w, b, h, 3 + c), DECODE_CHUNK, w.d, u, w.L + cs, pl)
            lo, hi = max(t0, cs), min(t0 + n, cs + DECODE_CHUNK)
            q[lo - t0:hi - t0, i] = _store(qq[lo - cs:hi - cs], w.dtype)
            k[lo - t0:hi - t0, i] = _store(kk[lo - cs:hi - cs], w.dtype)
            v[lo - t0:hi - t0, i] = _store(vv[lo - cs:hi - cs], w.dtype)

    if n > 0:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(one, range(len(hs))))
    return q, k, v


def as_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Storage form -> exact float64 values (what the oracle consumes)."""
    if dtype == "bf16":
        return bf16_bits_to_f32(x).astype(np.float64)
    return np.asarray(x, dtype=np.float32).astype(np.float64)


# ------------------------------------------------------------- exact ties
# A second recipe, for parity cases whose eviction and selection decisions
# are exact ties in fp32 as well as in fp64.  Every query is q = 8 e_0.  A
# "live" key has e_0 component 0 (its logit is exactly 0 under any rounding);
# a "dead" key has e_0 component -2048 (logit -2048 at d = 64, -1448 at
# d = 128), so its softmax weight underflows to exactly 0 next to any live
# key and its accumulated score stays exactly 0.  Dead entries therefore tie
# at score 0 and only the tie rule separates them.  Position 0 is always
# live, so every query attends to at least one live key.  The other
# components of keys, and all values, are N(0, 1).
TIE_Q = 8.0
TIE_DEAD = -2048.0
TIE_STREAM = 1 << 30


def _tie_rows(w: Workload, b: int, h: int, segment: int, first_pos: int, n: int, dead_frac: float):
    rng = np.random.default_rng([w.seed, b, h, TIE_STREAM, segment])  # apart from the main recipe's streams
    k = rng.standard_normal((n, w.d), dtype=np.float32)
    v = rng.standard_normal((n, w.d), dtype=np.float32)
    dead = rng.random(n) < dead_frac
    if first_pos == 0:
        dead[0] = False
    k[:, 0] = np.where(dead, np.float32(TIE_DEAD), np.float32(0.0))
    q = np.zeros((n, w.d), np.float32)
    q[:, 0] = TIE_Q
    return q, k, v


def tie_prompt(w: Workload, dead_frac: float, heads=None):
    """Prompt Q, K, V of the exact-tie recipe, like prompt()."""
    hs = _heads(w, heads)
    st = np.uint16 if w.dtype == "bf16" else np.float32
    Q = np.empty((len(hs), w.L, w.d), st)
    K = np.empty_like(Q)
    V = np.empty_like(Q)
    for i, f in enumerate(hs):
        b, h = divmod(f, w.H)
        q, k, v = _tie_rows(w, b, h, 0, 0, w.L, dead_frac)
        Q[i], K[i], V[i] = _store(q, w.dtype), _store(k, w.dtype), _store(v, w.dtype)
    return Q, K, V


def tie_decode(w: Workload, dead_frac: float, heads=None):
    """Decode inputs of all w.T steps of the exact-tie recipe, like decode()."""
    hs = _heads(w, heads)
    st = np.uint16 if w.dtype == "bf16" else np.float32
    q = np.empty((w.T, len(hs), w.d), st)
    k = np.empty_like(q)
    v = np.empty_like(q)
    for i, f in enumerate(hs):
        b, h = divmod(f, w.H)
        qq, kk, vv = _tie_rows(w, b, h, 1, w.L, w.T, dead_frac)
        q[:, i], k[:, i], v[:, i] = _store(qq, w.dtype), _store(kk, w.dtype), _store(vv, w.dtype)
    return q, k, v

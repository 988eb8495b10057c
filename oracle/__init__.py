"""ctypes front end of the fp64 CPU oracle (``h2o_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke``
and by the CPU-baseline leg of ``bench.py``.  The product path (the CUDA
library and its binding) never imports this package.

The oracle follows the H2O summary page ("The mechanism", "Algorithm /
figure walkthrough", Definition 4.3); see ``h2o_oracle.h`` for the readings
taken where the page is silent.  Parity pins: ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "h2o_oracle.c")
_LIB = os.path.join(_HERE, "libh2o_oracle.so")
_lib = None


def compile_source(src: str, out: str) -> str:
    """gcc, fp64, OpenMP, no fast-math, no FMA contraction (same results on
    x86-64 and aarch64)."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-I", _HERE,
                           "-fno-fast-math", "-ffp-contract=off", "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle if it is missing or older than its sources."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "h2o_oracle.h"))):
        compile_source(_SRC, _LIB)
    return _LIB


def load(path: str):
    """Load an oracle build (the default one, or another build of the same
    source for the tests' planted-mistake checks)."""
    L = C.CDLL(path)
    dp, ip = C.POINTER(C.c_double), C.POINTER(C.c_int32)
    L.h2o_oracle_prefill.argtypes = [C.c_int] * 8 + [dp] * 6 + [ip, dp, dp, dp, dp, dp, ip, dp, dp]
    L.h2o_oracle_prefill.restype = C.c_int
    L.h2o_oracle_decode.argtypes = [C.c_int] * 7 + [C.c_int64, C.c_int] + [ip, dp, dp, dp, dp, dp, ip] + \
        [dp] * 3 + [dp, ip, dp, dp]
    L.h2o_oracle_decode.restype = C.c_int
    L.h2o_oracle_set_threads.argtypes = [C.c_int]
    L.h2o_oracle_max_threads.restype = C.c_int
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = load(build())
    return _lib


def _p(a, ct=C.c_double):
    return None if a is None else a.ctypes.data_as(C.POINTER(ct))


def set_threads(n: int) -> None:
    lib().h2o_oracle_set_threads(int(n))


def max_threads() -> int:
    return int(lib().h2o_oracle_max_threads())


class State:
    """Oracle cache state of nh heads, k slots each (slot order carries no
    meaning: only the set of positions and their scores do)."""

    def __init__(self, nh: int, k: int, d: int):
        self.pos = np.full((nh, k), -1, np.int32)
        self.score = np.zeros((nh, k), np.float64)
        self.K = np.zeros((nh, k, d), np.float64)
        self.V = np.zeros((nh, k, d), np.float64)
        self.Ksc = np.ones((nh, k), np.float64)  # per-row scales of an fp8 cache
        self.Vsc = np.ones((nh, k), np.float64)
        self.n_valid = np.zeros(nh, np.int32)

    def copy(self) -> "State":
        s = State.__new__(State)
        s.pos, s.score, s.K, s.V, s.Ksc, s.Vsc, s.n_valid = (
            self.pos.copy(), self.score.copy(), self.K.copy(), self.V.copy(), self.Ksc.copy(),
            self.Vsc.copy(), self.n_valid.copy())
        return s

    def sets(self):
        """Sorted live positions of each head."""
        return [np.sort(p[p >= 0]) for p in self.pos]


def prefill(Q, K, V, k_heavy: int, k_local: int, _L=None, n_sink: int = 0, score_mode: int = 0,
            kv_fp8: bool = False):
    """Q, K, V: float64 [nh, L, d].  Returns dict with O, lse, colsum, state,
    margin, dropped_mass.  ``n_sink`` pins the first positions,
    ``score_mode`` 1 ranks by mean weight and ``kv_fp8`` stores cached rows
    as e4m3 with per-row scales (see ``h2o_oracle.h``)."""
    Q, K, V = (np.ascontiguousarray(x, np.float64) for x in (Q, K, V))
    nh, L, d = Q.shape
    k = k_heavy + k_local
    st = State(nh, k, d)
    O = np.empty((nh, L, d))
    lse = np.empty((nh, L))
    colsum = np.empty((nh, L))
    margin = np.empty(nh)
    dropped = np.empty(nh)
    rc = (_L or lib()).h2o_oracle_prefill(nh, d, L, k_heavy, k_local, n_sink, score_mode, int(kv_fp8), _p(Q),
                                          _p(K), _p(V), _p(O), _p(lse), _p(colsum), _p(st.pos, C.c_int32),
                                          _p(st.score), _p(st.K), _p(st.V), _p(st.Ksc), _p(st.Vsc),
                                          _p(st.n_valid, C.c_int32), _p(margin), _p(dropped))
    if rc != 0:
        raise ValueError("h2o_oracle_prefill: bad arguments")
    return dict(O=O, lse=lse, colsum=colsum, state=st, margin=margin, dropped_mass=dropped)


def decode(state: State, p0: int, q, k, v, k_heavy: int, k_local: int, want_out: bool = True,
           _L=None, n_sink: int = 0, score_mode: int = 0, kv_fp8: bool = False):
    """Run T decode steps in place on ``state``.  q, k, v: float64 [T, nh, d].
    Returns dict with out [T, nh, d], evicted [T, nh], margin [T, nh],
    evicted_mass [nh]."""
    q, k, v = (np.ascontiguousarray(x, np.float64) for x in (q, k, v))
    T, nh, d = q.shape
    out = np.empty((T, nh, d)) if want_out else None
    ev = np.empty((T, nh), np.int32)
    mg = np.empty((T, nh))
    em = np.zeros(nh)
    rc = (_L or lib()).h2o_oracle_decode(nh, d, k_heavy, k_local, n_sink, score_mode, int(kv_fp8), int(p0), T,
                                         _p(state.pos, C.c_int32), _p(state.score), _p(state.K), _p(state.V),
                                         _p(state.Ksc), _p(state.Vsc), _p(state.n_valid, C.c_int32),
                                         _p(q), _p(k), _p(v), _p(out), _p(ev, C.c_int32), _p(mg), _p(em))
    if rc != 0:
        raise ValueError("h2o_oracle_decode: bad arguments")
    return dict(out=out, evicted=ev, margin=mg, evicted_mass=em)

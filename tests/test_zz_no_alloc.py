"""h2o_decode_step_static: the decode step that allocates nothing.

Some callers cannot allocate device memory — servers that reserve all of HBM
up front and give a plugin only its input and output tensors, C hosts that
receive device pointers from another runtime, latency-critical loops that
cannot afford cudaMalloc — so this entry point keeps its scratch in a fixed
array inside the library.  Here it is called through the C ABI on two
consecutive decode steps and must reproduce the regular entry point
(h2o_decode_steps on a cache: the same evicted positions, cache sets, and
outputs and scores within the parity tolerances used elsewhere) and the fp64
oracle (outputs, evicted positions, cache sets and scores after each call).

This file is collected last on purpose (test_zz_*): it runs alone in a fresh
process as well as after every other test.
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import pytest
import torch

import h2o_heavy_hitter_decode_gb300 as h2o
import oracle
import synth
from h2o_heavy_hitter_decode_gb300 import H2OCache
from parity_helpers import MARGIN_TOL, SCORE_RTOL, out_atol, tdtype, to_dev

pytestmark = pytest.mark.gpu


def _entry():
    f = h2o.lib().h2o_decode_step_static
    f.argtypes = [C.c_int] * 6 + [C.c_void_p] * 4 + [C.c_int, C.c_int64] + [C.c_void_p] * 6
    f.restype = C.c_int
    return f


def _p(t):
    return C.c_void_p(t.data_ptr())


CASES = [
    synth.Workload("bf16_evicting", 2, 4, 128, 300, 2, 64, 64, "bf16", 4242),
    synth.Workload("f32_admitting", 1, 3, 64, 40, 2, 30, 20, "f32", 4243),
    synth.Workload("bf16_full_from_prefill", 3, 5, 64, 96, 2, 40, 24, "bf16", 4244),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_static_scratch_matches_regular_step(w):
    f = _entry()
    Qs, Ks, Vs = synth.prompt(w)
    qs, ks, vs = synth.decode(w, 0, 2)
    cache = H2OCache(w.B, w.H, w.d, w.k_heavy, w.k_local, tdtype(w))
    shp = (w.B, w.H, w.L, w.d)
    cache.prefill(to_dev(Qs, w, shp), to_dev(Ks, w, shp), to_dev(Vs, w, shp))
    st = cache.export()
    # The caller's own copy of the state, continued by the allocation-free call.
    K, V, pos, score = (st[x].clone() for x in ("K", "V", "pos", "score"))
    n_valid, position = st["n_valid"], st["next_pos"]
    dshp = (2, w.B, w.H, w.d)
    qd, kd, vd = to_dev(qs, w, dshp), to_dev(ks, w, dshp), to_dev(vs, w, dshp)
    stream = torch.cuda.current_stream()
    dt = 1 if w.dtype == "bf16" else 0
    cv = lambda x: synth.as_f64(x, w.dtype)
    o_st = oracle.prefill(cv(Qs), cv(Ks), cv(Vs), w.k_heavy, w.k_local)["state"]
    for t in range(2):  # two calls in a row on the same scratch
        ev_ref = torch.full((1, w.B, w.H), -7, dtype=torch.int32, device="cuda")
        ref = cache.steps(qd[t:t + 1], kd[t:t + 1], vd[t:t + 1], evicted=ev_ref)[0]
        od = oracle.decode(o_st, position, cv(qs[t:t + 1]), cv(ks[t:t + 1]), cv(vs[t:t + 1]), w.k_heavy,
                           w.k_local)
        out = torch.full_like(ref, float("nan"))
        ev = torch.full((w.B, w.H), -7, dtype=torch.int32, device="cuda")
        rc = f(w.B, w.H, w.d, w.k_heavy, w.k_local, dt, _p(K), _p(V), _p(pos), _p(score), n_valid, position,
               _p(qd[t]), _p(kd[t]), _p(vd[t]), _p(out), _p(ev), C.c_void_p(stream.cuda_stream))
        assert rc == 0, h2o.lib().h2o_status_str(rc)
        n_valid = min(n_valid + 1, w.k)
        position += 1
        torch.cuda.synchronize()
        err = (out.float() - ref.float()).abs().max().item()
        assert err <= out_atol(w.dtype), err
        assert torch.equal(ev, ev_ref[0]), "evicted positions differ from the regular step"
        # against the oracle: outputs, evicted positions (margins here are far
        # from the near-tie band), sets and scores
        o_err = float(np.abs(out.float().cpu().numpy().reshape(w.nh, w.d) - od["out"][0]).max())
        assert o_err <= out_atol(w.dtype), o_err
        assert np.all(od["margin"][0] > MARGIN_TOL), od["margin"][0]
        np.testing.assert_array_equal(ev.cpu().numpy().reshape(w.nh), od["evicted"][0])
        for h, o_set in enumerate(o_st.sets()):
            g_set = np.sort(pos.cpu().numpy().reshape(w.nh, w.k)[h])
            assert np.array_equal(g_set[g_set >= 0], o_set), f"step {t} head {h}: set differs from the oracle"
        g_sc = dict(zip(zip(np.repeat(np.arange(w.nh), w.k), pos.cpu().numpy().ravel()), score.cpu().numpy().ravel()))
        o_live = [(h, int(p_), float(s_)) for h in range(w.nh) for p_, s_ in zip(o_st.pos[h], o_st.score[h]) if p_ >= 0]
        rel = max(abs(g_sc[(h, p_)] - s_) / max(abs(s_), 1e-30) for h, p_, s_ in o_live)
        assert rel <= SCORE_RTOL, rel
        ref_state = cache.export()
        torch.cuda.synchronize()
        gp, rp = pos.cpu().numpy().reshape(w.nh, w.k), ref_state["pos"].cpu().numpy().reshape(w.nh, w.k)
        for h in range(w.nh):
            assert np.array_equal(np.sort(gp[h]), np.sort(rp[h])), f"step {t} head {h}: cache sets differ"
        gs = dict(zip(zip(np.repeat(np.arange(w.nh), w.k), gp.ravel()), score.cpu().numpy().ravel()))
        rs = dict(zip(zip(np.repeat(np.arange(w.nh), w.k), rp.ravel()), ref_state["score"].cpu().numpy().ravel()))
        live = [key for key in rs if key[1] >= 0]
        a = np.array([gs[key] for key in live], np.float64)
        b = np.array([rs[key] for key in live], np.float64)
        assert np.max(np.abs(a - b) / np.maximum(np.abs(b), 1e-30)) <= SCORE_RTOL
    assert cache.info()["n_valid"] == n_valid and cache.info()["next_pos"] == position


def test_static_scratch_rejects_oversized_shapes():
    f = _entry()
    x = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    i = torch.zeros(16, dtype=torch.int32, device="cuda")
    s = torch.zeros(16, dtype=torch.float32, device="cuda")
    # 64*56 heads x 8001 logits alone is far beyond the fixed scratch size.
    rc = f(64, 56, 128, 4000, 4001, 1, _p(x), _p(x), _p(i), _p(s), 0, 0, _p(x), _p(x), _p(x), _p(x), None,
           None)
    assert rc == 1  # H2O_EINVAL, nothing launched
    torch.cuda.synchronize()

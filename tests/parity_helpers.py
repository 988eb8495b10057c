"""GPU-vs-oracle parity harness shared by the GPU tests, the smoke check and
the bench's parity leg.

Tolerances (fixed by the method's acceptance rules):
  * cache sets: bit-exact; a mismatch is permitted only where the oracle's
    eviction margin (gap between the two lowest candidate ranking keys; for
    prefill the gap between the smallest kept and largest dropped key; the
    key is the score, or the mean weight under score_mode 1) is above 0 and
    at or below 1e-5, and it is then counted, the GPU is resynchronised from
    the oracle's state through h2o_cache_import, and the run continues.  At
    a margin of exactly 0 the tie rule (eviction: lowest position; prefill:
    the higher positions survive) makes the answer unique, so a mismatch
    there fails; such exact ties are counted (Report.ties_*);
  * attention outputs: max abs error <= 1e-4 (fp32 cache) or 2e-2 (bf16);
  * scores and column sums: relative error <= 1e-3;
  * lse: abs error <= 1e-4 (fp32 output in both cases);
  * fp8 caches: the stored e4m3 codes and row scales of every cached
    position are bit-exact (integer work: the same quantisation decisions).
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle
import synth
from h2o_heavy_hitter_decode_gb300 import H2OCache

MARGIN_TOL = 1e-5
SCORE_RTOL = 1e-3
LSE_ATOL = 1e-4
CHUNK = 256  # decode steps compared per round trip


def out_atol(dtype: str) -> float:
    return 1e-4 if dtype == "f32" else 2e-2


def tdtype(w):
    return torch.bfloat16 if w.dtype == "bf16" else torch.float32


def to_dev(x: np.ndarray, w, shape=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x.view(np.int16) if w.dtype == "bf16" else x))
    t = t.cuda()
    if w.dtype == "bf16":
        t = t.view(torch.bfloat16)
    return t.reshape(shape) if shape is not None else t


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def storage_from_f64(x: np.ndarray, w) -> np.ndarray:
    """Oracle K/V rows (exact copies of storage values) back to storage form."""
    x32 = x.astype(np.float32)
    return synth.f32_to_bf16_bits(x32) if w.dtype == "bf16" else x32


@dataclasses.dataclass
class Report:
    set_mismatch_prefill: int = 0
    set_mismatch_decode: int = 0
    resyncs: int = 0
    max_margin_at_mismatch: float = 0.0
    min_margin_seen: float = float("inf")
    max_out_err: float = 0.0
    max_O_err: float = 0.0
    max_lse_err: float = 0.0
    max_colsum_rel: float = 0.0
    max_score_rel: float = 0.0
    steps_compared: int = 0
    heads_compared: int = 0
    ties_prefill: int = 0  # heads whose prefill selection was an exact tie (oracle margin 0)
    ties_decode: int = 0   # (head, step) evictions that were exact ties, among the compared ones


def permitted(margin) -> bool:
    """A set mismatch is allowed only at a near-tie: 0 < margin <= 1e-5."""
    m = np.asarray(margin, dtype=np.float64)
    return bool(np.all((m > 0.0) & (m <= MARGIN_TOL)))


def _rel(a, b):
    return float(np.max(np.abs(a - b) / np.maximum(np.abs(b), 1e-30))) if a.size else 0.0


def fp8_codes(rows: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """e4m3 code values of oracle fp8 rows (row = code * scale exactly)."""
    sc = scale[..., None]
    return np.where(sc > 0, rows / np.where(sc > 0, sc, 1.0), 0.0)


def import_oracle_state(cache: H2OCache, st: oracle.State, w, next_pos: int):
    B, H, k, d = w.B, w.H, w.k, w.d
    pos = torch.from_numpy(st.pos.reshape(B, H, k).copy()).cuda()
    score = torch.from_numpy(st.score.astype(np.float32).reshape(B, H, k)).cuda()
    nv = int(st.n_valid[0])
    assert (st.n_valid == nv).all()
    if cache.kv_fp8:
        to8 = lambda x: torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).reshape(B, H, k, d).cuda()
        K, V = to8(fp8_codes(st.K, st.Ksc)), to8(fp8_codes(st.V, st.Vsc))
        ksc = torch.from_numpy(st.Ksc.astype(np.float32).reshape(B, H, k)).cuda()
        vsc = torch.from_numpy(st.Vsc.astype(np.float32).reshape(B, H, k)).cuda()
        cache.import_state(pos, score, K, V, next_pos, nv, ksc, vsc)
        return
    K = to_dev(storage_from_f64(st.K, w), w, (B, H, k, d))
    V = to_dev(storage_from_f64(st.V, w), w, (B, H, k, d))
    cache.import_state(pos, score, K, V, next_pos, nv)


def compare_fp8_rows(ex, o_st: oracle.State, heads, nh, k, d):
    """Stored codes and scales of every cached position, GPU vs oracle,
    bit-exact (slots matched by position)."""
    g_pos = ex["pos"].cpu().numpy().reshape(nh, k)
    gK = ex["K"].float().cpu().numpy().reshape(nh, k, d)
    gV = ex["V"].float().cpu().numpy().reshape(nh, k, d)
    gks = ex["K_scale"].cpu().numpy().reshape(nh, k)
    gvs = ex["V_scale"].cpu().numpy().reshape(nh, k)
    oK, oV = fp8_codes(o_st.K, o_st.Ksc), fp8_codes(o_st.V, o_st.Vsc)
    for i, h in enumerate(heads):
        gslot = {int(p): s for s, p in enumerate(g_pos[h]) if p >= 0}
        for s, p in enumerate(o_st.pos[i]):
            if p < 0:
                continue
            g = gslot[int(p)]
            assert gks[h, g] == np.float32(o_st.Ksc[i, s]) and gvs[h, g] == np.float32(o_st.Vsc[i, s]), (h, p)
            np.testing.assert_array_equal(gK[h, g], oK[i, s], err_msg=f"K codes head {h} pos {p}")
            np.testing.assert_array_equal(gV[h, g], oV[i, s], err_msg=f"V codes head {h} pos {p}")


def compare_scores(rep: Report, g_pos, g_score, o_st: oracle.State, heads):
    for i, h in enumerate(heads):
        gp, gs = g_pos[h], g_score[h]
        op, os_ = o_st.pos[i], o_st.score[i]
        gm = {int(p): float(s) for p, s in zip(gp, gs) if p >= 0}
        om = {int(p): float(s) for p, s in zip(op, os_) if p >= 0}
        assert set(gm) == set(om), f"head {h}: cache sets differ"
        keys = sorted(om)
        rep.max_score_rel = max(rep.max_score_rel, _rel(np.array([gm[p] for p in keys]), np.array([om[p] for p in keys])))


def run_parity(w, T=None, heads=None, resync=True, check=True, prompt=None, dec=None, want_O=True,
               decode_form="auto", policy=(0, 0), kv_fp8=False):
    """Prefill + T decode steps on the GPU through the C ABI, against the
    oracle on `heads` (all heads when None; resynchronisation needs all).
    `policy` = (n_sink, score_mode) of both sides; `kv_fp8` stores the cache
    rows as e4m3 with row scales on both sides."""
    T = w.T if T is None else T
    nh = w.nh
    hs = list(range(nh)) if heads is None else list(heads)
    all_heads = len(hs) == nh
    assert all_heads or not resync
    rep = Report(heads_compared=len(hs))
    Qs, Ks, Vs = prompt if prompt is not None else synth.prompt(w)

    cache = H2OCache(w.B, w.H, w.d, w.k_heavy, w.k_local, tdtype(w), kv_fp8=kv_fp8)
    cache.set_decode_form(decode_form)
    pol = dict(n_sink=policy[0], score_mode=policy[1], kv_fp8=kv_fp8)
    cache.set_policy(policy[0], policy[1])
    shp = (w.B, w.H, w.L, w.d)
    O, lse, colsum = cache.prefill(to_dev(Qs, w, shp), to_dev(Ks, w, shp), to_dev(Vs, w, shp), want_O=want_O)
    torch.cuda.synchronize()

    cv = lambda x: synth.as_f64(x, w.dtype)
    r = oracle.prefill(cv(Qs[hs]), cv(Ks[hs]), cv(Vs[hs]), w.k_heavy, w.k_local, **pol)
    if O is not None:
        rep.max_O_err = float(np.max(np.abs(f64(O).reshape(nh, w.L, w.d)[hs] - r["O"])))
    rep.max_lse_err = float(np.max(np.abs(f64(lse).reshape(nh, w.L)[hs] - r["lse"])))
    rep.max_colsum_rel = _rel(f64(colsum).reshape(nh, w.L)[hs], r["colsum"])
    if check:
        assert rep.max_O_err <= out_atol(w.dtype), rep
        assert rep.max_lse_err <= LSE_ATOL, rep
        assert rep.max_colsum_rel <= SCORE_RTOL, rep

    ex = cache.export()
    g_pos = ex["pos"].cpu().numpy().reshape(nh, w.k)
    st0 = r["state"]
    o_sets = st0.sets()
    bad = [i for i, h in enumerate(hs) if not np.array_equal(np.sort(g_pos[h][g_pos[h] >= 0]), o_sets[i])]
    rep.min_margin_seen = min(rep.min_margin_seen, float(np.min(r["margin"])))
    rep.ties_prefill = int(np.sum(r["margin"] == 0.0))
    if bad:
        rep.set_mismatch_prefill = len(bad)
        rep.max_margin_at_mismatch = max(rep.max_margin_at_mismatch, float(np.max(r["margin"][bad])))
        if check:
            assert permitted(r["margin"][bad]), (bad, r["margin"][bad])
        if resync:
            import_oracle_state(cache, st0, w, w.L)
            rep.resyncs += 1
    else:
        compare_scores(rep, g_pos, ex["score"].cpu().numpy().reshape(nh, w.k), st0, hs)
        if kv_fp8 and check:
            compare_fp8_rows(ex, st0, hs, nh, w.k, w.d)
    if T == 0:
        return rep, cache

    # Decode in chunks of CHUNK steps: the oracle advances its own state over
    # the chunk; the GPU runs the chunk through the C ABI and is compared step
    # by step (evicted position, output), resynchronised from the oracle after
    # a permitted near-tie divergence (resync mode) or dropped from the
    # comparison for the rest of the run (sampled-heads mode).
    o_st = st0.copy()
    alive = np.ones(len(hs), bool)
    if bad and not resync:
        alive[bad] = False
    hs_t = torch.tensor(hs, device="cuda")
    t0 = 0
    while t0 < T:
        n = min(CHUNK, T - t0)
        if dec is not None:
            qs, ks, vs = (x[t0:t0 + n] for x in dec)
        else:
            qs, ks, vs = synth.decode(w, t0, n)
        q64, k64, v64 = cv(qs[:, hs]), cv(ks[:, hs]), cv(vs[:, hs])
        st_start = o_st.copy()
        od = oracle.decode(o_st, w.L + t0, q64, k64, v64, w.k_heavy, w.k_local, **pol)
        o_ev, o_mg, o_out = od["evicted"], od["margin"], od["out"]
        finite = o_mg[:, alive][np.isfinite(o_mg[:, alive])]
        if finite.size:
            rep.min_margin_seen = min(rep.min_margin_seen, float(finite.min()))
        zero = (o_mg == 0.0)  # exact ties of this chunk (counted where compared)
        qd = to_dev(qs, w, (n, w.B, w.H, w.d))
        kd = to_dev(ks, w, (n, w.B, w.H, w.d))
        vd = to_dev(vs, w, (n, w.B, w.H, w.d))
        t = 0
        while t < n:
            m = n - t
            ev = torch.empty((m, w.B, w.H), dtype=torch.int32, device="cuda")
            out = cache.steps(qd[t:], kd[t:], vd[t:], evicted=ev)
            g_ev = ev.reshape(m, nh)[:, hs_t].cpu().numpy()
            g_out = f64(out.reshape(m, nh, w.d)[:, hs_t])
            diff = (g_ev != o_ev[t:]) & alive[None, :]
            if not resync:
                for i in np.nonzero(alive)[0]:
                    f = int(np.argmax(diff[:, i])) if diff[:, i].any() else m
                    upto = min(f + 1, m)
                    rep.max_out_err = max(rep.max_out_err, float(np.abs(g_out[:upto, i] - o_out[t:t + upto, i]).max()))
                    rep.ties_decode += int(np.sum(zero[t:t + upto, i]))
                    if f < m:
                        alive[i] = False
                        rep.set_mismatch_decode += 1
                        rep.max_margin_at_mismatch = max(rep.max_margin_at_mismatch, float(o_mg[t + f, i]))
                        if check:
                            assert permitted(o_mg[t + f, i]), (t0 + t + f, hs[i], o_mg[t + f, i])
                rep.steps_compared += m
                break
            first = int(np.argmax(diff.any(1))) if diff.any() else m
            upto = min(first + 1, m)  # the divergent step's output is still comparable
            rep.max_out_err = max(rep.max_out_err, float(np.abs(g_out[:upto] - o_out[t:t + upto]).max()))
            rep.steps_compared += upto
            rep.ties_decode += int(np.sum(zero[t:t + upto]))
            if first == m:
                break
            cols = np.nonzero(diff[first])[0]
            mg = o_mg[t + first, cols]
            rep.set_mismatch_decode += len(cols)
            rep.max_margin_at_mismatch = max(rep.max_margin_at_mismatch, float(mg.max()))
            if check:
                assert permitted(mg), (t0 + t + first, [hs[c] for c in cols], mg)
            st = st_start.copy()
            oracle.decode(st, w.L + t0, q64[:t + first + 1], k64[:t + first + 1], v64[:t + first + 1],
                          w.k_heavy, w.k_local, want_out=False, **pol)
            import_oracle_state(cache, st, w, w.L + t0 + t + first + 1)
            rep.resyncs += 1
            t = t + first + 1
        t0 += n
    if check:
        assert rep.max_out_err <= out_atol(w.dtype), rep
    ex = cache.export()
    torch.cuda.synchronize()
    g_pos = ex["pos"].cpu().numpy().reshape(nh, w.k)
    g_sc = ex["score"].cpu().numpy().reshape(nh, w.k)
    sel = [i for i in range(len(hs)) if alive[i]]
    if sel:
        sub = oracle.State(len(sel), w.k, w.d)
        sub.pos, sub.score = o_st.pos[sel], o_st.score[sel]
        compare_scores(rep, g_pos, g_sc, sub, [hs[i] for i in sel])
        if kv_fp8 and check:
            sub.K, sub.V, sub.Ksc, sub.Vsc = o_st.K[sel], o_st.V[sel], o_st.Ksc[sel], o_st.Vsc[sel]
            compare_fp8_rows(ex, sub, [hs[i] for i in sel], nh, w.k, w.d)
    if check:
        assert rep.max_score_rel <= SCORE_RTOL, rep
        cache.check_device_error()
    return rep, cache

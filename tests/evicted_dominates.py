"""Decode inputs under which the entry just evicted would take most of the
next query's attention.

The pipelined decode form runs step t+1's attention pass over the cache as it
was before step t's decision and then removes the evicted entry's term from
its partial sums.  When that term is most of the partial mass the removal
would cancel catastrophically, so the kernel recomputes the partial instead.
These inputs make that case common: after every `every`-th step t the oracle
reports the evicted position e_t, and q_{t+1} is set to point along K at e_t,
scaled so that q_{t+1} . K_e / sqrt(d) = beta.  The oracle, run step by step,
fixes the evictions; nothing here depends on the GPU path."""
from __future__ import annotations

import numpy as np

import oracle
import synth


def build(w, every: int = 2, beta: float = 20.0, kv_fp8: bool = False, policy=(0, 0)):
    """Returns (prompt, dec, dominated): synth-format prompt and decode inputs
    of workload w, and how many (step, head) pairs have the evicted entry
    holding more than half of the next query's softmax mass over the cache it
    was evicted from."""
    Qs, Ks, Vs = synth.prompt(w)
    qs, ks, vs = synth.decode(w, 0, w.T)
    q = qs.copy()
    cv = lambda x: synth.as_f64(x, w.dtype)
    pol = dict(n_sink=policy[0], score_mode=policy[1], kv_fp8=kv_fp8)
    st = oracle.prefill(cv(Qs), cv(Ks), cv(Vs), w.k_heavy, w.k_local, **pol)["state"]
    dominated = 0
    for t in range(w.T):
        K0, pos0 = st.K.copy(), st.pos.copy()
        od = oracle.decode(st, w.L + t, cv(q[t:t + 1]), cv(ks[t:t + 1]), cv(vs[t:t + 1]), w.k_heavy, w.k_local,
                           want_out=False, **pol)
        if t + 1 >= w.T or t % every:
            continue
        for h in range(w.nh):
            e = int(od["evicted"][0, h])
            if e < 0 or e == w.L + t:
                continue
            s = int(np.nonzero(pos0[h] == e)[0][0])
            ke = K0[h, s]
            nn = float(ke @ ke)
            if nn == 0.0:
                continue
            qn = (beta * np.sqrt(w.d) / nn) * ke
            q[t + 1, h] = synth.f32_to_bf16_bits(qn.astype(np.float32)) if w.dtype == "bf16" else qn.astype(np.float32)
            qv = cv(q[t + 1, h])
            live = pos0[h] >= 0
            lg = K0[h][live] @ qv / np.sqrt(w.d)
            share = np.exp(lg[np.nonzero(pos0[h][live] == e)[0][0]] - lg.max()) / np.exp(lg - lg.max()).sum()
            dominated += int(share > 0.5)
    return (Qs, Ks, Vs), (q, ks, vs), dominated

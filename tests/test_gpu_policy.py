"""GPU parity of the eviction policy variants (pinned attention sinks and
mean-weight ranking, h2o_cache_set_policy) against the fp64 oracle run with
the same policy, through the C ABI, every decode form; tolerances as in
parity_helpers."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import synth
from h2o_heavy_hitter_decode_gb300 import H2OCache, H2OError
from parity_helpers import run_parity

pytestmark = pytest.mark.gpu

W = synth.Workload


def small(name, B, H, d, L, T, kh, kl, dt, seed=91, planted=0.0):
    return W(name, B, H, d, L, T, kh, kl, dt, seed, planted)


# (workload, [(n_sink, score_mode), ...]); n_sink = k_heavy is sinks + window
CASES = [
    (synth.TINY, [(4, 0), (0, 1), (4, 1), (16, 0)]),
    (small("bf16_multitile_ragged", 2, 3, 128, 300, 40, 64, 64, "bf16"), [(8, 0), (0, 1), (8, 1), (64, 0)]),
    (small("bf16_no_local_block", 1, 2, 128, 100, 50, 32, 0, "bf16"), [(4, 1), (32, 0)]),
    (small("bf16_d64_prompt_shorter_than_budget", 1, 4, 64, 50, 80, 40, 30, "bf16"), [(10, 1)]),
    (small("bf16_planted_hitters", 2, 2, 128, 257, 64, 30, 30, "bf16", planted=0.05), [(4, 1), (0, 1)]),
    (small("f32_many_heads_splits", 4, 8, 64, 200, 24, 50, 40, "f32"), [(6, 1)]),
]
PARAMS = [(w, pol) for w, pols in CASES for pol in pols]


@pytest.mark.parametrize("form", ["per_step", "cooperative", "cluster", "pipelined"])
@pytest.mark.parametrize("w,policy", PARAMS, ids=[f"{w.name}-sink{p[0]}-mode{p[1]}" for w, p in PARAMS])
def test_policy_all_heads(w, policy, form):
    rep, cache = run_parity(w, decode_form=form, policy=policy)
    print(w.name, policy, form, rep)
    assert rep.steps_compared >= w.T
    assert cache.policy() == tuple(policy)
    if policy[0] > 0:  # the sinks are still cached
        pos = cache.export()["pos"].cpu().numpy().reshape(w.nh, w.k)
        for h in range(w.nh):
            assert set(range(min(policy[0], w.L + w.T))) <= set(pos[h].tolist())


def _sample(w, count, seed=5):
    rng = np.random.default_rng(seed)
    return sorted(rng.choice(w.nh, size=min(count, w.nh), replace=False).tolist())


@pytest.mark.parametrize("w,count,policy", [(synth.OPT_6_7B, 8, (4, 1)), (synth.OPT_6_7B, 8, (256, 0)),
                                            (synth.OPT_30B, 8, (0, 1))],
                         ids=lambda x: getattr(x, "name", str(x)))
def test_policy_full_size_sampled_heads(w, count, policy):
    """Full-size workloads in the bench's launch configuration (automatic
    decode form) on a seeded head sample."""
    rep, cache = run_parity(w, heads=_sample(w, count), resync=False, policy=policy)
    print(w.name, policy, rep)
    assert rep.steps_compared >= w.T


def test_policy_arguments_rejected():
    c = H2OCache(1, 2, 64, 8, 8, torch.bfloat16)
    for ns, mode in [(-1, 0), (9, 0), (0, 2), (0, -1)]:
        with pytest.raises(H2OError):
            c.set_policy(ns, mode)
    assert c.policy() == (0, 0)
    c.set_policy(8, 1)
    assert c.policy() == (8, 1)

"""GPU parity of the fp8 K/V cache (H2O_BF16_FP8KV: e4m3 codes, one fp32
scale per row) against the fp64 oracle run with the same storage rule,
through the C ABI and every decode form.  Stored codes and scales are
compared bit-exactly; outputs, scores and sets as for bf16 (parity_helpers)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import synth
from h2o_heavy_hitter_decode_gb300 import H2OCache, H2OError
from parity_helpers import run_parity, to_dev

pytestmark = pytest.mark.gpu

W = synth.Workload


def small(name, B, H, d, L, T, kh, kl, seed=123, planted=0.0):
    return W(name, B, H, d, L, T, kh, kl, "bf16", seed, planted)


CASES = [
    small("fp8_multitile_ragged", 2, 3, 128, 300, 40, 64, 64),
    small("fp8_d64_prompt_shorter_than_budget", 1, 4, 64, 50, 80, 40, 30),
    small("fp8_no_local_block", 1, 2, 128, 100, 50, 32, 0),
    small("fp8_single_token_prompt", 1, 2, 64, 1, 20, 4, 4),
    small("fp8_k1_heavy", 1, 2, 128, 40, 20, 1, 0),
    small("fp8_planted_hitters", 2, 2, 128, 257, 64, 30, 30, planted=0.05),
    small("fp8_many_heads_long_budget", 4, 6, 128, 700, 40, 200, 100),
]


@pytest.mark.parametrize("form", ["per_step", "cooperative", "cluster", "pipelined"])
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_fp8_all_heads(w, form):
    rep, cache = run_parity(w, decode_form=form, kv_fp8=True)
    print(w.name, form, rep)
    assert rep.steps_compared >= w.T


@pytest.mark.parametrize("form", ["per_step", "cluster", "pipelined"])
def test_fp8_with_policy(form):
    w = small("fp8_sinks_mean", 2, 3, 128, 300, 40, 64, 64)
    rep, cache = run_parity(w, decode_form=form, kv_fp8=True, policy=(8, 1))
    print(w.name, form, rep)
    assert rep.steps_compared >= w.T


@pytest.mark.parametrize("w", [small("fp8_cluster_long_chunks_resident", 1, 2, 128, 2600, 24, 1300, 1100),
                               small("fp8_d64_cluster_long_chunks_resident", 1, 2, 64, 2500, 24, 1200, 1200)],
                         ids=lambda w: w.name)
@pytest.mark.parametrize("form", ["cluster", "pipelined"])
def test_fp8_cluster_long_chunks(w, form):
    """300 fp8 slots per cluster CTA: their rows (77 KB or 38 KB of codes) stay
    resident in shared memory and four consumer warps read them."""
    rep, cache = run_parity(w, decode_form=form, kv_fp8=True)
    print(w.name, form, rep)
    assert cache.decode_form_used() == form
    assert -(-w.k // min(cache.info()["n_split"], 8)) > 256  # slots per CTA
    assert rep.steps_compared >= w.T


def _sample(w, count, seed=5):
    rng = np.random.default_rng(seed)
    return sorted(rng.choice(w.nh, size=min(count, w.nh), replace=False).tolist())


@pytest.mark.parametrize("w,count", [(synth.OPT_6_7B, 8), (synth.OPT_30B, 8), (synth.PREFILL_HEAVY, 2)],
                         ids=lambda x: getattr(x, "name", str(x)))
def test_fp8_full_size_sampled_heads(w, count):
    """Full-size workloads with an fp8 cache in the bench's launch
    configuration (automatic decode form) on a seeded head sample."""
    rep, cache = run_parity(w, heads=_sample(w, count), resync=False, kv_fp8=True)
    print(w.name, rep)
    assert rep.steps_compared >= w.T


def test_fp8_long_stream_first_steps():
    w = synth.LONG_STREAM
    rep, cache = run_parity(w, T=8192, kv_fp8=True)
    print(w.name, rep)
    assert rep.steps_compared >= 8192


def test_fp8_export_import_continues_identically():
    """A second cache imported from the first's exported codes and scales
    continues with identical outputs and state."""
    w = small("fp8_roundtrip", 1, 4, 128, 200, 24, 48, 32)
    Q, K, V = synth.prompt(w)
    shp = (w.B, w.H, w.L, w.d)
    a = H2OCache(w.B, w.H, w.d, w.k_heavy, w.k_local, torch.bfloat16, kv_fp8=True)
    a.prefill(to_dev(Q, w, shp), to_dev(K, w, shp), to_dev(V, w, shp))
    q, k, v = (to_dev(x, w, (w.T, w.B, w.H, w.d)) for x in synth.decode(w, 0, w.T))
    a.steps(q[:8], k[:8], v[:8])
    ex = a.export()
    b = H2OCache(w.B, w.H, w.d, w.k_heavy, w.k_local, torch.bfloat16, kv_fp8=True)
    b.import_state(ex["pos"], ex["score"], ex["K"], ex["V"], ex["next_pos"], ex["n_valid"], ex["K_scale"],
                   ex["V_scale"])
    oa = a.steps(q[8:], k[8:], v[8:])
    ob = b.steps(q[8:], k[8:], v[8:])
    torch.cuda.synchronize()
    assert torch.equal(oa, ob)
    ea, eb = a.export(), b.export()
    for key in ("pos", "score", "K_scale", "V_scale"):
        assert torch.equal(ea[key], eb[key]), key
    assert torch.equal(ea["K"].view(torch.uint8), eb["K"].view(torch.uint8))
    assert torch.equal(ea["V"].view(torch.uint8), eb["V"].view(torch.uint8))


def test_scales_unsupported_on_bf16_cache():
    from h2o_heavy_hitter_decode_gb300 import lib
    c = H2OCache(1, 2, 64, 8, 8, torch.bfloat16)
    assert lib().h2o_cache_export_scales(c._h, None, None) == 6
    with pytest.raises(TypeError):
        H2OCache(1, 2, 64, 8, 8, torch.float32, kv_fp8=True)

"""Prefill by batch rows (h2o_prefill_rows): groups of rows prefilled in any
order give bit-identical outputs, cache state and decode to one whole-batch
prefill (heads are independent and each kernel works per head)."""
from __future__ import annotations

import pytest
import torch

import synth
from h2o_heavy_hitter_decode_gb300 import H2OCache, H2OError
from parity_helpers import to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kv_fp8", [False, True])
def test_rows_match_whole_prefill(kv_fp8):
    w = synth.Workload("rows_bf16_B4H3", 4, 3, 128, 300, 24, 48, 32, "bf16", 321)
    Q, K, V = synth.prompt(w)
    shp = (w.B, w.H, w.L, w.d)
    Qd, Kd, Vd = to_dev(Q, w, shp), to_dev(K, w, shp), to_dev(V, w, shp)
    q, k, v = (to_dev(x, w, (w.T, w.B, w.H, w.d)) for x in synth.decode(w, 0, w.T))

    whole = H2OCache(w.B, w.H, w.d, w.k_heavy, w.k_local, torch.bfloat16, kv_fp8=kv_fp8)
    O1, l1, c1 = whole.prefill(Qd, Kd, Vd)
    rows = H2OCache(w.B, w.H, w.d, w.k_heavy, w.k_local, torch.bfloat16, kv_fp8=kv_fp8)
    O2, l2, c2 = torch.empty_like(O1), torch.empty_like(l1), torch.empty_like(c1)
    for b0, nb in [(2, 2), (0, 1), (1, 1)]:  # out of order, uneven groups
        sl = slice(b0, b0 + nb)
        o, l, c = rows.prefill_rows(b0, Qd[sl].contiguous(), Kd[sl].contiguous(), Vd[sl].contiguous())
        O2[sl], l2[sl], c2[sl] = o, l, c
    torch.cuda.synchronize()
    assert torch.equal(O1, O2) and torch.equal(l1, l2) and torch.equal(c1, c2)
    e1, e2 = whole.export(), rows.export()
    for key in e1:
        if isinstance(e1[key], torch.Tensor):
            assert torch.equal(e1[key].view(torch.uint8), e2[key].view(torch.uint8)), key
        else:
            assert e1[key] == e2[key], key
    assert torch.equal(whole.steps(q, k, v), rows.steps(q, k, v))
    whole.check_device_error()
    rows.check_device_error()


def test_rows_state_rules():
    w = synth.Workload("rows_rules", 2, 2, 64, 40, 4, 8, 8, "bf16", 322)
    Q, K, V = synth.prompt(w)
    shp = (w.B, w.H, w.L, w.d)
    Qd, Kd, Vd = to_dev(Q, w, shp), to_dev(K, w, shp), to_dev(V, w, shp)
    q, k, v = (to_dev(x, w, (1, w.B, w.H, w.d)) for x in synth.decode(w, 0, 1))
    c = H2OCache(w.B, w.H, w.d, w.k_heavy, w.k_local, torch.bfloat16)
    c.prefill_rows(0, Qd[:1].contiguous(), Kd[:1].contiguous(), Vd[:1].contiguous())
    with pytest.raises(H2OError):  # decode before every row is prefilled
        c.steps(q, k, v)
    with pytest.raises(H2OError):  # the same row twice
        c.prefill_rows(0, Qd[:1].contiguous(), Kd[:1].contiguous(), Vd[:1].contiguous())
    with pytest.raises(H2OError):  # another prompt length
        c.prefill_rows(1, Qd[1:, :, :32].contiguous(), Kd[1:, :, :32].contiguous(), Vd[1:, :, :32].contiguous())
    with pytest.raises(H2OError):  # rows past B
        c.prefill_rows(1, Qd.contiguous(), Kd.contiguous(), Vd.contiguous())
    c.prefill_rows(1, Qd[1:].contiguous(), Kd[1:].contiguous(), Vd[1:].contiguous())
    c.steps(q, k, v)
    torch.cuda.synchronize()
    c.check_device_error()

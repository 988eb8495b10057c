#!/usr/bin/env python
"""Benchmark of the H2O decode/prefill hot path on GB300.

One bench step = one whole job of the workload: create the cache, prefill the
prompt (causal attention + column sums + heavy-hitter selection), then T
decode steps (attend, accumulate scores, evict, write in place), all through
the C ABI with inputs already resident in HBM.  L2 is flushed (a 256 MB write)
before every step, outside the timed events.

Printed JSON line (rank 0):
  value     generated tokens/s of the whole job (B*T per job, per layer),
            summed over ranks (weak scaling: each rank runs its own job);
  decode    decode-only tokens/s, KV-read GB/s and fractions of HBM peak;
  prefill   score-pass (column sums) and attention-pass TFLOP/s;
  roofline  the kernel with the largest share of the step, measured live with
            CUDA events on the launching stream (the C ABI's phase timer);
  e2e       the same metric with host (pinned) buffers, copies timed;
  cpu_baseline  the fp64 oracle on the host cores on a sample of heads.

`--impl reference` times the oracle alone (the reference arm: the method's
reference semantics on the host cores).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

NOMINAL_HBM_GBS = 8000.0
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
METRIC = "H2O decode tokens/s and KV-read GB/s vs HBM peak; prefill score TFLOP/s"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {k: float(d[k]) for k in FALLBACK}, "measured"
    return dict(FALLBACK), "fallback"


FP8_SUFFIX = "_kvfp8"  # workload name suffix of a run with an fp8 K/V cache (--kv fp8)


def is_kvfp8(w):
    return w.name.endswith(FP8_SUFFIX)


def esize(w):
    """Bytes per input / output element."""
    return 2 if w.dtype == "bf16" else 4


def slot_kv_bytes(w):
    """Stored K+V bytes of one cache slot: two rows, plus two fp32 row scales
    for an fp8 cache."""
    return 2 * w.d + 8 if is_kvfp8(w) else 2 * w.d * esize(w)


def decode_alg_bytes(w):
    """Algorithmic HBM bytes of one decode step: K and V slots, position tags,
    score read+write, the step's q/k/v inputs and its output."""
    return w.nh * (w.k * slot_kv_bytes(w) + 12 * w.k) + 4 * w.nh * w.d * esize(w)


def kv_read_bytes(w):
    return w.nh * w.k * slot_kv_bytes(w)


def score_pass_flops(w):
    """Causal QK^T of the column-sum pass: d*L*(L+1) per head."""
    return w.nh * w.d * w.L * (w.L + 1)


def attn_pass_flops(w):
    return 2 * score_pass_flops(w)


def causal_exps(w):
    """One exponential per causal (query, key) pair in each prefill pass."""
    return w.nh * w.L * (w.L + 1) // 2


EX2_PER_CLK_PER_SM = 32  # ex2.approx.f32 issue rate, measured on GB300 with a register-resident loop


def workload_config(w, extra=None):
    c = {"workload": w.name, "B": w.B, "H": w.H, "d": w.d, "prompt_L": w.L, "decode_T": w.T,
         "k_heavy": w.k_heavy, "k_local": w.k_local,
         "cache_dtype": "e4m3 + fp32 row scale" if is_kvfp8(w) else w.dtype,
         "global_batch": w.B, "seq_len": w.L + w.T, "parallelism": "none (heads independent)",
         "l2": "flushed before every step (256 MB write)"}
    if extra:
        c.update(extra)
    return c


def src_sha(rel):
    return hashlib.sha256(open(os.path.join(ROOT, rel), "rb").read()).hexdigest()[:16]


def traffic_for(kernel, w):
    """DRAM bytes per launch of `kernel` on workload `w` from a committed ncu
    capture, or None if none was taken or the kernel source changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(f"{kernel}@{w.name}")
    if not d:
        return None
    if d.get("source_sha") != src_sha(d["source"]):
        return None
    return d.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks

class Clocks:
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"h2o_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            return self
        # nvidia-smi takes a moment to start: let its first sample land before
        # the timed region begins, so the samples cover that region
        t_end = time.time() + 3.0
        while time.time() < t_end and self.proc.poll() is None:
            self.f.flush()
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 8:
                try:
                    rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[4:8]))
                except ValueError:
                    pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = np.array([r[0] for r in rows])
        load = sm[sm > 0.5 * sm.max()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median(load)), "sm_max_mhz": float(rows[0][1]), "reasons": reasons,
                "samples": len(rows), "power_w_max": float(max(r[2] for r in rows))}


# ------------------------------------------------------------ multi-rank

def aggregate_over_ranks(total_ms, steps, tokens_per_job, world, dist=None, device="cpu"):
    """Whole-job figures of a weak-scaling run: every rank times its own job;
    the slowest rank's total time counts, and the value is the tokens of all
    ranks' jobs over that time.  Returns (ms_per_step, tokens_per_s)."""
    if dist is not None and world > 1:
        import torch
        t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_per_step = total_ms / steps
    return ms_per_step, tokens_per_job * world / (ms_per_step / 1e3)


# --------------------------------------------------------------- our arm

def run_ours(args, w, rank, world, local_rank):
    import torch
    import h2o_heavy_hitter_decode_gb300 as h2o
    from h2o_heavy_hitter_decode_gb300 import H2OCache
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    else:
        torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    h2o.lib()
    pk, pk_src = peaks()

    Qs, Ks, Vs = synth.prompt(w)
    qs, ks, vs = synth.decode(w, 0, w.T)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    def host(x, shape):
        t = torch.from_numpy(np.ascontiguousarray(x.view(np.int16) if w.dtype == "bf16" else x))
        if w.dtype == "bf16":
            t = t.view(torch.bfloat16)
        return t.reshape(shape)

    shp_p, shp_d = (w.B, w.H, w.L, w.d), (w.T, w.B, w.H, w.d)
    hQ, hK, hV = host(Qs, shp_p), host(Ks, shp_p), host(Vs, shp_p)
    hq, hk, hv = host(qs, shp_d), host(ks, shp_d), host(vs, shp_d)
    Qd, Kd, Vd, qd, kd, vd = (x.to(dev) for x in (hQ, hK, hV, hq, hk, hv))
    O = torch.empty(shp_p, dtype=tdt, device=dev)
    lse = torch.empty((w.B, w.H, w.L), dtype=torch.float32, device=dev)
    colsum = torch.empty_like(lse)
    out = torch.empty(shp_d, dtype=tdt, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def job():
        c = H2OCache(w.B, w.H, w.d, w.k_heavy, w.k_local, tdt, device=dev, kv_fp8=is_kvfp8(w))
        c.set_decode_form(args.decode_form)
        c.profile(True)
        c.prefill(Qd, Kd, Vd, O=O, lse=lse, colsum=colsum)
        c.steps(qd, kd, vd, out=out)
        return c

    for _ in range(args.warmup):
        flush.zero_()
        job().profile_read()
    torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    phases = {p: [0.0, 0] for p in H2OCache.PHASES}
    caches = []
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with Clocks(local_rank) as clk:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            caches.append(job())
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    if dist:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    for c in caches:
        for p, (ms, n) in c.profile_read().items():
            phases[p][0] += ms
            phases[p][1] += n
    caches[-1].check_device_error()
    K = args.steps
    ms_per_step, value = aggregate_over_ranks(float(np.sum(step_ms)), K, w.B * w.T, world, dist, dev)

    dec_ms = phases["decode"][0] / K
    dec_launch_ms = dec_ms / w.T  # per decode step (a multi-step form runs many steps per launch)
    form = caches[-1].decode_form_used()
    dec_kernel = {"cluster": "decode_cluster_kernel", "cooperative": "decode_kernel",
                  "per_step": "decode_kernel"}.get(form, "decode_kernel")
    kv_gbs = kv_read_bytes(w) / (dec_launch_ms / 1e3) / 1e9
    dec_alg_gbs = decode_alg_bytes(w) / (dec_launch_ms / 1e3) / 1e9
    cs_ms = phases["prefill_colsum"][0] / K
    at_ms = phases["prefill_attn"][0] / K
    sel_ms = phases["prefill_select"][0] / K
    cs_tf = score_pass_flops(w) / (cs_ms / 1e3) / 1e12
    at_tf = attn_pass_flops(w) / (at_ms / 1e3) / 1e12

    clk_sum = clk.summary()
    sm_mhz = clk_sum.get("sm_mhz") or clk_sum.get("sm_max_mhz")
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count

    def exp_rate(ms):  # exponentials per SM clock per SM over the pass
        return causal_exps(w) / (ms / 1e3 * sm_mhz * 1e6 * n_sms) if sm_mhz else None

    shares = {"decode": dec_ms, "prefill_colsum": cs_ms, "prefill_attn": at_ms, "prefill_select": sel_ms}
    top = max(shares, key=shares.get)
    if top == "decode":
        roof = {"kernel": dec_kernel, "decode_form": form, "bound": "hbm", "achieved": dec_alg_gbs,
                "peak": pk["hbm_gbs"], "unit": "GB/s", "traffic": traffic_for(dec_kernel, w),
                "per": "decode step (algorithmic bytes and DRAM traffic per step)",
                "algorithmic_bytes_per_launch": decode_alg_bytes(w), "avg_launch_ms": dec_launch_ms,
                "cache_in_l2": kv_read_bytes(w) < 120e6}
        if roof["cache_in_l2"]:
            roof["note"] = ("the K/V cache fits in L2 and stays there across steps, so the steps read it from L2 "
                            "(see traffic: DRAM bytes per step); the fraction is of the HBM copy bandwidth")
    elif top == "prefill_colsum":
        roof = {"kernel": "prefill_colsum", "bound": "tensor", "achieved": cs_tf, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "traffic": traffic_for("prefill_colsum", w),
                "per": "launch", "algorithmic_flops_per_launch": score_pass_flops(w), "avg_launch_ms": cs_ms}
    else:
        roof = {"kernel": top, "bound": "tensor", "achieved": at_tf if top == "prefill_attn" else None,
                "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "traffic": traffic_for(top, w),
                "per": "launch", "algorithmic_flops_per_launch": attn_pass_flops(w), "avg_launch_ms": shares[top]}
    roof["frac"] = (roof["achieved"] / roof["peak"]) if roof.get("achieved") else None
    roof["peak_source"] = pk_src
    roof["share_of_step"] = shares[top] / ms_per_step

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "impl": "ours",
        "dtype_note": "stored K/V and tensor-core operands in this type; accumulation, softmax and scores in fp32",
        "data": "synthetic: seeded per-head generator (Pareto-shifted keys along a hidden direction)",
        "config": workload_config(w, {"decode_form": args.decode_form}),
        "decode": {"form": form, "tokens_per_s": w.B * world / (dec_launch_ms / 1e3), "us_per_step": dec_launch_ms * 1e3,
                   "kv_read_gbs": kv_gbs, "alg_gbs": dec_alg_gbs,
                   "kv_read_frac_measured_hbm": kv_gbs / pk["hbm_gbs"],
                   "kv_read_frac_nominal_8tbs": kv_gbs / NOMINAL_HBM_GBS,
                   "cache_bytes": kv_read_bytes(w), "l2_resident": kv_read_bytes(w) < 120e6},
        "prefill": {"score_pass_tflops": cs_tf, "score_pass_frac_measured_bf16": cs_tf / pk["bf16_tflops"],
                    "attn_pass_tflops": at_tf, "attn_pass_frac_measured_bf16": at_tf / pk["bf16_tflops"],
                    "ms": {"attn": at_ms, "colsum": cs_ms, "select_gather": sel_ms},
                    "exp_per_clk_per_sm": {"score_pass": exp_rate(cs_ms), "attn_pass": exp_rate(at_ms),
                                           "ex2_unit": EX2_PER_CLK_PER_SM, "sm_mhz": sm_mhz, "sms": n_sms}},
        "phase_ms_per_step": shares,
        "roofline": roof,
        "gpu_launches": int(phases["prefill_attn"][1] + phases["prefill_colsum"][1] + phases["prefill_select"][1]
                            + phases["decode"][1]),
        "wall_s_timed": t_wall,
        "clocks": clk_sum,
        "peaks": {**pk, "source": pk_src},
    }

    if not args.no_e2e:
        line["e2e"] = e2e(args, w, dev, hQ, hK, hV, hq, hk, hv, tdt, stream, world, dist,
                          row_groups=args.e2e_row_groups, step_groups=args.e2e_step_groups)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args)
    if dist:
        dist.destroy_process_group()
    return line if rank == 0 else None


def e2e(args, w, dev, hQ, hK, hV, hq, hk, hv, tdt, stream, world, dist, row_groups=8, step_groups=4):
    """Same job from pinned host buffers: H2D of every input, prefill, decode,
    D2H of the decode outputs, all inside the timed events.  The prompt is
    copied on a side stream in `row_groups` groups of batch rows and each
    group is prefilled (h2o_prefill_rows) as soon as it has landed, so the
    prefill of one group overlaps the copy of the next.  The decode inputs
    follow in `step_groups` groups of steps; each group is decoded as soon as
    its inputs have landed and its outputs are copied back while the next
    group decodes."""
    import torch
    from h2o_heavy_hitter_decode_gb300 import H2OCache
    pin = [x.pin_memory() for x in (hQ, hK, hV, hq, hk, hv)]
    dbuf = [torch.empty_like(x, device=dev) for x in pin]
    O = torch.empty(hQ.shape, dtype=tdt, device=dev)
    lse = torch.empty((w.B, w.H, w.L), dtype=torch.float32, device=dev)
    colsum = torch.empty_like(lse)
    out = torch.empty(hq.shape, dtype=tdt, device=dev)
    hout = torch.empty(hq.shape, dtype=tdt).pin_memory()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    side = torch.cuda.Stream(device=dev)
    back = torch.cuda.Stream(device=dev)
    ng = max(1, min(row_groups, w.B))
    groups = [(w.B * g // ng, w.B * (g + 1) // ng) for g in range(ng)]
    ns = max(1, min(step_groups, w.T))
    sgroups = [(w.T * g // ns, w.T * (g + 1) // ns) for g in range(ns)]

    def job(start_ev):
        side.wait_event(start_ev)
        landed = []
        with torch.cuda.stream(side):
            for b0, b1 in groups:  # prompt rows, group by group
                for t in (0, 1, 2):
                    dbuf[t][b0:b1].copy_(pin[t][b0:b1], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(side)
                landed.append(ev)
            dec_landed = []
            for t0, t1 in sgroups:  # decode inputs, behind the prompt, group by group
                for t in (3, 4, 5):
                    dbuf[t][t0:t1].copy_(pin[t][t0:t1], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(side)
                dec_landed.append(ev)
        c = H2OCache(w.B, w.H, w.d, w.k_heavy, w.k_local, tdt, device=dev, kv_fp8=is_kvfp8(w))
        c.set_decode_form(args.decode_form)
        for (b0, b1), ev in zip(groups, landed):
            stream.wait_event(ev)
            c.prefill_rows(b0, dbuf[0][b0:b1], dbuf[1][b0:b1], dbuf[2][b0:b1], O=O[b0:b1], lse=lse[b0:b1],
                           colsum=colsum[b0:b1])
        for (t0, t1), ev in zip(sgroups, dec_landed):
            stream.wait_event(ev)
            c.steps(dbuf[3][t0:t1], dbuf[4][t0:t1], dbuf[5][t0:t1], out=out[t0:t1])
            done = torch.cuda.Event()
            done.record(stream)
            back.wait_event(done)
            with torch.cuda.stream(back):
                hout[t0:t1].copy_(out[t0:t1], non_blocking=True)
        stream.wait_stream(back)  # the job ends when its outputs are on the host
        return c

    n = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(max(1, min(args.warmup, 3)) + n)]
    for i in range(max(1, min(args.warmup, 3))):
        ev[i][0].record(stream)
        job(ev[i][0])
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    timed = ev[len(ev) - n:]
    for a, b in timed:
        flush.zero_()
        a.record(stream)
        job(a)
        b.record(stream)
    torch.cuda.synchronize()
    ms_step, value = aggregate_over_ranks(float(np.sum([a.elapsed_time(b) for a, b in timed])), n, w.B * w.T,
                                          world, dist, dev)
    h2d = sum(x.numel() * x.element_size() for x in pin)
    d2h = hout.numel() * hout.element_size()
    return {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms_step, "prompt_row_groups": ng, "decode_step_groups": ns}


# ------------------------------------------------------------ oracle timing

CPU_SAMPLE_STEPS = 65536  # decode steps of the oracle sample (the long stream's first 65,536)


def oracle_sample(w, n_heads):
    """Inputs of the first n_heads heads and the first CPU_SAMPLE_STEPS
    decode steps (a bounded sample of the workload): (heads, steps, data)."""
    hs = list(range(min(n_heads, w.nh)))
    T = min(w.T, CPU_SAMPLE_STEPS)
    Q, K, V = (synth.as_f64(x, w.dtype) for x in synth.prompt(w, heads=hs))
    q, k, v = (synth.as_f64(x, w.dtype) for x in synth.decode(w, 0, T, heads=hs))
    return hs, T, (Q, K, V, q, k, v)


def sample_text(w, hs, T):
    return (f"{len(hs)} of {w.nh} heads, prefill L={w.L} + "
            + (f"{T} decode steps (the full job)" if T == w.T else f"the first {T} of {w.T} decode steps")
            + ("" if len(hs) == w.nh else "; rate extrapolated linearly to all heads"))


def oracle_job(w, data):
    """Wall-clock seconds of one oracle job on the sample: (prefill, decode)."""
    import oracle
    Q, K, V, q, k, v = data
    t0 = time.perf_counter()
    r = oracle.prefill(Q, K, V, w.k_heavy, w.k_local, kv_fp8=is_kvfp8(w))
    t1 = time.perf_counter()
    oracle.decode(r["state"], w.L, q, k, v, w.k_heavy, w.k_local, kv_fp8=is_kvfp8(w))
    return t1 - t0, time.perf_counter() - t1


CPU_SAMPLE_HEADS = 256  # the whole default workload; seconds of work on a many-core host


def cpu_baseline(w, args):
    import oracle
    cores = os.cpu_count() or 1
    oracle.set_threads(cores)
    hs, T, data = oracle_sample(w, CPU_SAMPLE_HEADS)
    pre, dec = oracle_job(w, data)
    secs = pre + dec
    scale = w.nh / len(hs)
    return {"value": w.B * T / (secs * scale), "unit": "tokens/s", "cores": int(oracle.max_threads()),
            "kind": "oracle", "phases_s": {"prefill": pre, "decode": dec},
            "sample": f"{sample_text(w, hs, T)}, {secs:.2f} s"}


def run_reference(args, w):
    import oracle
    cores = os.cpu_count() or 1
    oracle.set_threads(cores)
    hs, T, data = oracle_sample(w, CPU_SAMPLE_HEADS)
    for _ in range(args.warmup):
        oracle_job(w, data)
    phases = np.array([oracle_job(w, data) for _ in range(args.steps)])
    scale = w.nh / len(hs)
    per_job = float(np.mean(phases.sum(axis=1))) * scale
    value = w.B * T / per_job
    sample = f"each step: {sample_text(w, hs, T)}"
    return {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": per_job * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "impl": "reference",
            "data": "synthetic: seeded per-head generator", "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": int(oracle.max_threads()),
                             "kind": "oracle", "sample": sample,
                             "phases_s": {"prefill": float(np.mean(phases[:, 0])),
                                          "decode": float(np.mean(phases[:, 1]))}},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=1, help="workload index (0 tiny, 1 OPT-6.7B-shaped, ...)")
    ap.add_argument("--prompt-len", type=int, default=None, help="override L (profiling captures)")
    ap.add_argument("--decode-steps", type=int, default=None, help="override T (profiling captures)")
    ap.add_argument("--decode-form", default="auto", choices=["auto", "per_step", "cooperative", "cluster"])
    ap.add_argument("--kv", choices=["native", "fp8"], default="native",
                    help="K/V cache storage: the workload's dtype, or e4m3 codes with a row scale (bf16 workloads)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-row-groups", type=int, default=8, help="prompt row groups copied/prefilled in turn")
    ap.add_argument("--e2e-step-groups", type=int, default=4, help="decode step groups copied/decoded in turn")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    w = synth.CONFIGS[args.config]
    if args.prompt_len is not None or args.decode_steps is not None:
        L = w.L if args.prompt_len is None else args.prompt_len
        T = w.T if args.decode_steps is None else args.decode_steps
        w = w.with_(name=f"{w.name}[L={L},T={T}]", L=L, T=T)
    if args.kv == "fp8":
        if w.dtype != "bf16":
            ap.error("--kv fp8 needs a bf16 workload")
        w = w.with_(name=w.name + FP8_SUFFIX)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, w)), flush=True)
        return
    line = run_ours(args, w, rank, world, local_rank)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Benchmark of the H2O decode/prefill hot path on GB300.

One bench step = one whole job of the workload: create the cache, prefill the
prompt (causal attention + column sums + heavy-hitter selection), then T
decode steps (attend, accumulate scores, evict, write in place), all through
the C ABI with inputs already resident in HBM.  L2 is flushed (a 256 MB write)
before every job, outside the timed events; a job's decode steps then run back
to back, so a cache smaller than L2 is served from L2 after its first step
(the line says so: `decode.l2_resident`, `roofline.bound` "l2").

The default workload is the largest single-GPU one: the 8K-prompt serving
shape (B=32, H=32, d=128, L=8192, 256 decode steps, k = 845 + 845), whose
886 MB cache is read from HBM every step.  `--config N` picks another.

Printed JSON line (rank 0):
  value     generated tokens/s of the whole job (global batch x T per job,
            per layer, each token counted once, over the slowest rank's time);
  decode    decode-only tokens/s, KV-read GB/s and fractions of HBM peak;
  prefill   score-pass (column sums) and attention-pass TFLOP/s;
  roofline  the kernel with the largest share of the step, measured live with
            CUDA events on the launching stream (the C ABI's phase timer);
  e2e       the same metric with host (pinned) buffers, copies timed (for
            long prompts one cache per row group, each decoded as soon as
            its rows are prefilled, so the compute overlaps the host link);
  cpu_baseline  the fp64 oracle on the host cores on a bounded sample of heads.

Several GPUs: one process per GPU (torchrun, or `--gpus N`, which starts
torchrun itself).  The batch rows are sharded over the ranks with no exchange
between them (heads are independent): by default each rank runs B rows of a
global batch of N*B rows (`--scaling weak`); `--scaling strong` splits the
workload's B rows over the ranks instead.

The long stream (`--config 4`, 4,194,304 decode steps) is generated on the
device before the timed region (103 GB of inputs, resident in HBM) and decoded
in calls of 65,536 steps into a reused output buffer.

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
L2_RESIDENT_BYTES = 120e6  # caches below this stay in the 129 MB L2 across decode steps
METRIC = "H2O decode tokens/s and KV-read GB/s vs HBM peak; prefill score TFLOP/s"
DEFAULT_CONFIG = 3  # the 8K-prompt serving shape: the largest single-GPU workload
STREAM_CHUNK = 65536  # decode steps per call when the inputs are generated on the device
# The end-to-end leg pipelines by rows (prompt row groups prefilled as they
# land into a few caches, each decoded once its rows are prefilled) when each
# cache still holds this many heads: its decode grid then fills the GPU.
# Measured on GB300 (ms per job, one cache whose decode waits for every row /
# rows into 2 caches): 8K prompt 57.3 / 52.1, OPT-30B shape 100.9 / 90.3;
# OPT-6.7B shape (128 heads per cache) 5.75 / 8.12.
E2E_ROWS_MIN_HEADS = 512


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


def streamed(w):
    """Decode inputs too many for the host: generated on the device."""
    return w.T > STREAM_CHUNK


EX2_PER_CLK_PER_SM = 32  # ex2.approx.f32 issue rate, measured on GB300 with a register-resident loop


def workload_config(w, extra=None):
    c = {"workload": w.name, "B": w.B, "H": w.H, "d": w.d, "prompt_L": w.L, "decode_T": w.T,
         "k_heavy": w.k_heavy, "k_local": w.k_local,
         "cache_dtype": "e4m3 + fp32 row scale" if is_kvfp8(w) else w.dtype,
         "global_batch": w.B, "seq_len": w.L + w.T, "parallelism": "none (heads independent)",
         "l2": "flushed before every job (256 MB write); the decode steps of a job run back to back"}
    if extra:
        c.update(extra)
    return c


def src_sha(rel):
    return hashlib.sha256(open(os.path.join(ROOT, rel), "rb").read()).hexdigest()[:16]


def traffic_for(kernel, w):
    """DRAM bytes per launch of `kernel` on workload `w` from a committed ncu
    capture (profiles/traffic.json), with where it came from; (None, reason)
    if none was taken or the kernel source changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None, "no stored capture"
    d = json.load(open(p)).get(f"{kernel}@{w.name}")
    if not d:
        return None, f"no stored capture of {kernel} on this workload"
    if d.get("source_sha") != src_sha(d["source"]):
        return None, f"{d['source']} changed since the stored capture"
    how = d.get("capture", "ncu dram__bytes_read.sum + dram__bytes_write.sum")
    return d.get("dram_bytes_per_launch"), f"profiles/traffic.json ({how}; source {d['source']} @ {d['source_sha']})"


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

def rank_rows(B, world, rank, scaling="weak"):
    """Batch rows of one rank: (first global row, rows, global batch).

    weak: every rank runs B rows of a global batch of world*B rows (rank r
    owns rows r*B .. r*B+B-1), so the work per GPU is fixed as ranks are
    added.  strong: the B rows are split over the ranks in contiguous,
    near-equal ranges.  Either way the ranges cover the global batch exactly
    once."""
    if scaling == "weak":
        return rank * B, B, B * world
    if scaling != "strong":
        raise ValueError(f"scaling must be 'weak' or 'strong', not {scaling!r}")
    if world > B:
        raise ValueError(f"strong scaling needs at least one batch row per rank (B={B}, ranks={world})")
    b0, b1 = B * rank // world, B * (rank + 1) // world
    return b0, b1 - b0, B


def aggregate_over_ranks(total_ms, steps, tokens_total, world, dist=None, device="cpu"):
    """Whole-job figures of a multi-rank run: every rank times its own share;
    the slowest rank's total time counts, and the value is the tokens of all
    ranks' shares (each counted once, `tokens_total`) over that time.
    Returns (ms_per_step, tokens_per_s)."""
    if dist is not None and world > 1:
        import torch
        t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_per_step = total_ms / steps
    return ms_per_step, tokens_total / (ms_per_step / 1e3)


def relaunch_under_torchrun(n):
    """`--gpus n` without a process group: start n ranks with torchrun on
    this node and return their exit status."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


# ------------------------------------------------------- device-side inputs

def device_decode_inputs(w, t0, n, heads, dev, out):
    """Decode inputs of steps t0 .. t0+n-1 for `heads` generated on the device
    into out = (q, k, v), each [n, len(heads), d]: the workload's recipe (the
    head's unit direction u from synth, keys N(0,I) + s u with s Type-I
    Pareto(1.5) clipped to 8, queries N(0,I) + 2u, values N(0,1)) drawn from
    torch's counter-based generator seeded per (workload, step range), then
    rounded once to the storage type.  Not bit-identical to synth.decode (a
    different random stream); used where the host cannot hold the inputs."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(int(w.seed) * 1000003 + int(t0))
    u = torch.from_numpy(np.stack([synth._direction(w, *divmod(h, w.H)) for h in heads])).to(dev)
    nh, d = len(heads), w.d
    kn = torch.randn((n, nh, d), generator=g, device=dev)
    uni = torch.rand((n, nh), generator=g, device=dev, dtype=torch.float64)
    s = torch.clamp((1.0 - uni) ** (-1.0 / synth.PARETO_ALPHA), max=synth.PARETO_CLIP).float()
    out[1].copy_(kn.add_(s[:, :, None] * u[None]))
    del kn
    qn = torch.randn((n, nh, d), generator=g, device=dev)
    out[0].copy_(qn.add_(synth.QUERY_SHIFT * u[None]))
    del qn
    out[2].copy_(torch.randn((n, nh, d), generator=g, device=dev))


def l2_read_gbs(dev, nbytes):
    """Read bandwidth of an L2-resident buffer the size of the K/V cache
    (clamped to 16..96 MB), measured here with the library's read kernel
    (h2o_probe_read, 16-byte loads through L2): the roof of a decode step
    whose cache stays in L2 (the step only reads it)."""
    import h2o_heavy_hitter_decode_gb300 as h2o
    n = int(min(max(nbytes, 16 << 20), 96 << 20))
    return h2o.probe_read_gbs(n, reps=100, device=dev), n


# --------------------------------------------------------------- our arm

def run_ours(args, w, rank, world, local_rank):
    import torch
    import h2o_heavy_hitter_decode_gb300 as h2o
    from h2o_heavy_hitter_decode_gb300 import H2OCache
    dist = None
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    dev = torch.device("cuda", local_rank)
    h2o.lib()
    pk, pk_src = peaks()

    # This rank's batch rows of the global batch; inputs are generated for
    # those global rows (seeded by row), so every rank runs distinct data.
    b0, nb, Bg = rank_rows(w.B, world, rank, args.scaling)
    wg = w.with_(B=Bg)
    wl = w.with_(B=nb)
    heads = list(range(b0 * w.H, (b0 + nb) * w.H))
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    def host(x, shape):
        t = torch.from_numpy(np.ascontiguousarray(x.view(np.int16) if w.dtype == "bf16" else x))
        if w.dtype == "bf16":
            t = t.view(torch.bfloat16)
        return t.reshape(shape)

    shp_p, shp_d = (nb, w.H, w.L, w.d), (w.T, nb, w.H, w.d)
    Qs, Ks, Vs = synth.prompt(wg, heads=heads)
    hQ, hK, hV = host(Qs, shp_p), host(Ks, shp_p), host(Vs, shp_p)
    del Qs, Ks, Vs
    if streamed(w):
        chunk = STREAM_CHUNK
        qd, kd, vd = (torch.empty(shp_d, dtype=tdt, device=dev) for _ in range(3))
        for t0 in range(0, w.T, chunk):
            n = min(chunk, w.T - t0)
            device_decode_inputs(wg, t0, n, heads, dev,
                                 tuple(x[t0:t0 + n].view(n, nb * w.H, w.d) for x in (qd, kd, vd)))
        out = torch.empty((chunk, nb, w.H, w.d), dtype=tdt, device=dev)
        hq = hk = hv = None
    else:
        chunk = w.T
        qs, ks, vs = synth.decode(wg, 0, w.T, heads=heads)
        hq, hk, hv = host(qs, shp_d), host(ks, shp_d), host(vs, shp_d)
        del qs, ks, vs
        qd, kd, vd = (x.to(dev) for x in (hq, hk, hv))
        out = torch.empty(shp_d, dtype=tdt, device=dev)
    Qd, Kd, Vd = (x.to(dev) for x in (hQ, hK, hV))
    O = torch.empty(shp_p, dtype=tdt, device=dev)
    lse = torch.empty((nb, w.H, w.L), dtype=torch.float32, device=dev)
    colsum = torch.empty_like(lse)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def job():
        c = H2OCache(nb, w.H, w.d, w.k_heavy, w.k_local, tdt, device=dev, kv_fp8=is_kvfp8(w))
        c.set_decode_form(args.decode_form)
        c.profile(True)
        c.prefill(Qd, Kd, Vd, O=O, lse=lse, colsum=colsum)
        for t0 in range(0, w.T, chunk):
            n = min(chunk, w.T - t0)
            c.steps(qd[t0:t0 + n], kd[t0:t0 + n], vd[t0:t0 + n], out=out[:n])
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
    ms_per_step, value = aggregate_over_ranks(float(np.sum(step_ms)), K, Bg * w.T, world, dist, dev)

    dec_ms = phases["decode"][0] / K
    dec_launch_ms = dec_ms / w.T  # per decode step (a multi-step form runs many steps per launch)
    form = caches[-1].decode_form_used()
    dec_kernel = {"cluster": "decode_cluster_kernel", "pipelined": "decode_pipe_kernel",
                  "cooperative": "decode_kernel", "per_step": "decode_kernel"}.get(form, "decode_kernel")
    kv_gbs = kv_read_bytes(wl) / (dec_launch_ms / 1e3) / 1e9
    dec_alg_gbs = decode_alg_bytes(wl) / (dec_launch_ms / 1e3) / 1e9
    cs_ms = phases["prefill_colsum"][0] / K
    at_ms = phases["prefill_attn"][0] / K
    sel_ms = phases["prefill_select"][0] / K
    cs_tf = score_pass_flops(wl) / (cs_ms / 1e3) / 1e12
    at_tf = attn_pass_flops(wl) / (at_ms / 1e3) / 1e12
    in_l2 = kv_read_bytes(wl) < L2_RESIDENT_BYTES  # the whole cache fits in L2

    clk_sum = clk.summary()
    sm_mhz = clk_sum.get("sm_mhz") or clk_sum.get("sm_max_mhz")
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count

    def exp_rate(ms):  # exponentials per SM clock per SM over the pass
        return causal_exps(wl) / (ms / 1e3 * sm_mhz * 1e6 * n_sms) if sm_mhz else None

    shares = {"decode": dec_ms, "prefill_colsum": cs_ms, "prefill_attn": at_ms, "prefill_select": sel_ms}
    top = max(shares, key=shares.get)
    # Where the decode's bytes come from: the stored DRAM traffic of this kernel
    # on this workload (when its source is unchanged since the capture) shows
    # whether the steps read the cache from L2 (e.g. the cluster form's waves,
    # each smaller than L2, run all their steps before the next wave); without
    # a capture, whether the whole cache fits in L2.
    dec_traffic, dec_traffic_src = traffic_for(dec_kernel, w)
    if dec_traffic is not None and world == 1:
        l2_served = dec_traffic < 0.5 * decode_alg_bytes(wl)
        served_how = (f"stored capture: {dec_traffic / 1e6:.1f} MB of DRAM traffic per step against "
                      f"{decode_alg_bytes(wl) / 1e6:.1f} MB of algorithmic bytes")
    else:
        l2_served = in_l2
        served_how = "the whole cache " + ("fits" if in_l2 else "does not fit") + " in L2 (no matching traffic capture)"
    l2_gbs, l2_buf = l2_read_gbs(dev, kv_read_bytes(wl)) if l2_served else (None, 0)
    if top == "decode":
        roof = {"kernel": dec_kernel, "decode_form": form, "achieved": dec_alg_gbs, "unit": "GB/s",
                "traffic": dec_traffic, "traffic_source": dec_traffic_src,
                "per": "decode step (algorithmic bytes and DRAM traffic per step)",
                "algorithmic_bytes_per_launch": decode_alg_bytes(wl), "avg_launch_ms": dec_launch_ms,
                "cache_in_l2": in_l2, "served_from": "l2" if l2_served else "hbm", "served_from_evidence": served_how}
        if l2_served:
            roof.update(bound="l2", peak=l2_gbs, peak_source=(
                f"measured in this run: the library read kernel (h2o_probe_read) over an L2-resident {l2_buf / 1e6:.0f} MB buffer"),
                note="the decode steps read the K/V cache from L2, so the roof is L2 read bandwidth, not HBM")
        else:
            roof.update(bound="hbm", peak=pk["hbm_gbs"], peak_source=pk_src + " HBM copy bandwidth")
    elif top == "prefill_colsum":
        traffic, traffic_src = traffic_for("colsum_pair_tc", w)
        roof = {"kernel": "colsum_pair_tc", "bound": "tensor", "achieved": cs_tf, "peak": pk["bf16_tflops"],
                "peak_source": pk_src + " bf16 burst", "unit": "TFLOP/s", "traffic": traffic,
                "traffic_source": traffic_src, "per": "launch",
                "algorithmic_flops_per_launch": score_pass_flops(wl), "avg_launch_ms": cs_ms}
    else:
        kname = "attn_pair_tc" if top == "prefill_attn" else "select_gather"
        traffic, traffic_src = traffic_for(kname, w)
        roof = {"kernel": kname, "bound": "tensor",
                "achieved": at_tf if top == "prefill_attn" else None, "peak": pk["bf16_tflops"],
                "peak_source": pk_src + " bf16 burst", "unit": "TFLOP/s", "traffic": traffic,
                "traffic_source": traffic_src, "per": "launch",
                "algorithmic_flops_per_launch": attn_pass_flops(wl), "avg_launch_ms": shares[top]}
    roof["frac"] = (roof["achieved"] / roof["peak"]) if roof.get("achieved") and roof.get("peak") else None
    roof["share_of_step"] = shares[top] / ms_per_step

    decode = {"form": form, "tokens_per_s": Bg / (dec_launch_ms / 1e3), "us_per_step": dec_launch_ms * 1e3,
              "kv_read_gbs": kv_gbs, "alg_gbs": dec_alg_gbs, "cache_bytes": kv_read_bytes(wl),
              "l2_resident": in_l2, "served_from": "l2" if l2_served else "hbm", "served_from_evidence": served_how}
    if l2_served:
        decode.update(l2_read_gbs=l2_gbs, kv_read_frac_l2_read=kv_gbs / l2_gbs,
                      note="cache read from L2: a fraction of HBM bandwidth would overstate the kernel")
    else:
        decode.update(kv_read_frac_measured_hbm=kv_gbs / pk["hbm_gbs"],
                      kv_read_frac_nominal_8tbs=kv_gbs / NOMINAL_HBM_GBS)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": args.scaling,
        "vs_baseline": None, "dtype": w.dtype, "impl": "ours",
        "dtype_note": "stored K/V and tensor-core operands in this type; accumulation, softmax and scores in fp32",
        "data": "synthetic: seeded per-head generator (Pareto-shifted keys along a hidden direction)"
                + ("; decode inputs generated on the device" if streamed(w) else ""),
        "config": workload_config(w, {"decode_form": args.decode_form, "global_batch": Bg,
                                      "rows_per_rank": nb,
                                      "parallelism": (f"dp{world}: batch rows sharded over ranks, no exchange"
                                                      if world > 1 else "none (heads independent)")}),
        "decode": decode,
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
    if streamed(w):
        line["long_stream"] = long_stream_report(caches[-1], w, dec_launch_ms)

    del qd, kd, vd, Qd, Kd, Vd, O, out  # device inputs of the resident runs: room for the e2e buffers
    caches.clear()
    if not args.no_e2e:
        rows = args.e2e_pipeline == "rows" or (
            args.e2e_pipeline == "auto" and wl.B * w.H // max(1, args.e2e_decode_groups) >= E2E_ROWS_MIN_HEADS)
        if rows and not streamed(w):
            line["e2e"] = e2e_row_caches(args, w, wl, Bg, dev, hQ, hK, hV, hq, hk, hv, tdt, stream, world, dist,
                                         row_groups=args.e2e_row_groups, decode_groups=args.e2e_decode_groups)
        else:
            line["e2e"] = e2e(args, w, wl, Bg, heads, dev, hQ, hK, hV, hq, hk, hv, tdt, stream, world, dist,
                              row_groups=args.e2e_row_groups, step_groups=args.e2e_step_groups)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args)
    if dist:
        dist.destroy_process_group()
    return line if rank == 0 else None


def long_stream_report(cache, w, dec_step_ms):
    """Scores at the end of the stream: the largest one and its fp32 spacing,
    which bounds how finely later weights still register in it."""
    ex = cache.export()
    sc = ex["score"].float().cpu().numpy()
    pos = ex["pos"].cpu().numpy()
    live = sc[pos >= 0]
    smax = float(live.max())
    return {"decode_steps": w.T, "us_per_step": dec_step_ms * 1e3, "max_score": smax,
            "max_score_ulp": float(np.spacing(np.float32(smax))),
            "median_score": float(np.median(live)), "n_positions_seen": w.L + w.T,
            "score_mass_live": float(live.sum() / w.nh)}


def e2e(args, w, wl, Bg, heads, dev, hQ, hK, hV, hq, hk, hv, tdt, stream, world, dist, row_groups=8,
        step_groups=4):
    """Same job from pinned host buffers: H2D of every input, prefill, decode,
    D2H of the decode outputs, all inside the timed events.  The prompt is
    copied on a side stream in `row_groups` groups of batch rows and each
    group is prefilled (h2o_prefill_rows) as soon as it has landed, so the
    prefill of one group overlaps the copy of the next.  The decode inputs
    follow in `step_groups` groups of steps; each group is decoded as soon as
    its inputs have landed and its outputs are copied back while the next
    group decodes.  For device-generated decode inputs (the long stream) the
    host holds one chunk of STREAM_CHUNK steps, copied in for every chunk."""
    import torch
    from h2o_heavy_hitter_decode_gb300 import H2OCache
    nb = wl.B
    if streamed(w):
        shp = (STREAM_CHUNK, nb, w.H, w.d)
        gen = tuple(torch.empty(shp, dtype=tdt, device=dev) for _ in range(3))
        device_decode_inputs(w.with_(B=Bg), 0, STREAM_CHUNK, heads, dev,
                             tuple(x.view(STREAM_CHUNK, nb * w.H, w.d) for x in gen))
        hq, hk, hv = (x.cpu() for x in gen)
        del gen
        n_chunks = -(-w.T // STREAM_CHUNK)
        step_groups = n_chunks
    pin = [x.pin_memory() for x in (hQ, hK, hV, hq, hk, hv)]
    dbuf = [torch.empty_like(x, device=dev) for x in pin]
    O = torch.empty(hQ.shape, dtype=tdt, device=dev)
    lse = torch.empty((nb, w.H, w.L), dtype=torch.float32, device=dev)
    colsum = torch.empty_like(lse)
    out = torch.empty(hq.shape, dtype=tdt, device=dev)
    hout = torch.empty(hq.shape, dtype=tdt).pin_memory()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    side = torch.cuda.Stream(device=dev)
    back = torch.cuda.Stream(device=dev)
    ng = max(1, min(row_groups, nb))
    groups = [(nb * g // ng, nb * (g + 1) // ng) for g in range(ng)]
    if streamed(w):  # one chunk of host inputs per call, copied again for every chunk
        sgroups = [(0, min(STREAM_CHUNK, w.T - c * STREAM_CHUNK)) for c in range(step_groups)]
    else:
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
        c = H2OCache(nb, w.H, w.d, w.k_heavy, w.k_local, tdt, device=dev, kv_fp8=is_kvfp8(w))
        c.set_decode_form(args.decode_form)
        for (b0, b1), ev in zip(groups, landed):
            stream.wait_event(ev)
            c.prefill_rows(b0, dbuf[0][b0:b1], dbuf[1][b0:b1], dbuf[2][b0:b1], O=O[b0:b1], lse=lse[b0:b1],
                           colsum=colsum[b0:b1])
        for t0, t1 in sgroups:  # decode inputs behind the prompt, group by group
            with torch.cuda.stream(side):
                if streamed(w):  # one reused chunk buffer: refill it after the previous chunk's decode
                    side.wait_stream(stream)
                for t in (3, 4, 5):
                    dbuf[t][t0:t1].copy_(pin[t][t0:t1], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(side)
            stream.wait_event(ev)
            if streamed(w):  # one reused output buffer: after the previous chunk's copy back
                stream.wait_stream(back)
            c.steps(dbuf[3][t0:t1], dbuf[4][t0:t1], dbuf[5][t0:t1], out=out[t0:t1])
            done = torch.cuda.Event()
            done.record(stream)
            back.wait_event(done)
            with torch.cuda.stream(back):
                hout[t0:t1].copy_(out[t0:t1], non_blocking=True)
        stream.wait_stream(back)  # the job ends when its outputs are on the host
        return c

    # the host link alone: every input copied once from pinned memory, nothing else running
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for t in range(6):
        dbuf[t].copy_(pin[t], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    h2d_alone_ms = e0.elapsed_time(e1)
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
    ms_step, value = aggregate_over_ranks(float(np.sum([a.elapsed_time(b) for a, b in timed])), n, Bg * w.T,
                                          world, dist, dev)
    h2d_prompt = sum(x.numel() * x.element_size() for x in pin[:3])
    h2d_dec = sum(pin[t][t0:t1].numel() * pin[t].element_size() for t in (3, 4, 5) for t0, t1 in sgroups)
    d2h = sum(hout[t0:t1].numel() * hout.element_size() for t0, t1 in sgroups)
    all_in = sum(x.numel() * x.element_size() for x in pin)
    r = {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": h2d_prompt + h2d_dec, "d2h_bytes_per_step": d2h,
         "ms_per_step": ms_step, "prompt_row_groups": ng, "decode_step_groups": len(sgroups),
         "h2d_alone": {"ms": h2d_alone_ms, "gbs": all_in / (h2d_alone_ms / 1e3) / 1e9,
                       "what": "one copy of every input buffer from pinned host memory, nothing else running"}}
    if streamed(w):
        r["note"] = (f"decode inputs copied chunk by chunk from one pinned host chunk of {STREAM_CHUNK} steps "
                     "(the host cannot hold the whole stream's inputs)")
    return r


def e2e_row_caches(args, w, wl, Bg, dev, hQ, hK, hV, hq, hk, hv, tdt, stream, world, dist, row_groups=8,
                   decode_groups=2):
    """Same job from pinned host buffers, pipelined by batch rows: the batch is
    split into `decode_groups` caches (every head is independent, so the
    arithmetic is the same as one cache over all rows), each filled by
    `row_groups` / `decode_groups` prompt row groups.  A side stream copies
    the row groups' prompts in turn, and each cache's decode inputs after its
    last row group; the compute stream prefills each row group into its cache
    (h2o_prefill_rows) as soon as its rows have landed and decodes a cache as
    soon as all its rows are prefilled, while later rows are still crossing
    the host link; a cache's outputs copy back while later caches compute.
    Caches of several row groups keep the decode grids large.  The host
    buffers are laid out per group (contiguous rows) before the timed region."""
    import torch
    from h2o_heavy_hitter_decode_gb300 import H2OCache
    nb = wl.B
    nd = max(1, min(decode_groups, nb))
    caches_rows = [(nb * c // nd, nb * (c + 1) // nd) for c in range(nd)]
    per = max(1, row_groups // nd)  # prompt row groups per cache
    groups = []  # (cache index, first row, end row)
    for ci, (c0, c1) in enumerate(caches_rows):
        m = max(1, min(per, c1 - c0))
        groups += [(ci, c0 + (c1 - c0) * g // m, c0 + (c1 - c0) * (g + 1) // m) for g in range(m)]
    ng = len(groups)
    pin_p = [[x[b0:b1].contiguous().pin_memory() for x in (hQ, hK, hV)] for _, b0, b1 in groups]
    pin_d = [[x[:, c0:c1].contiguous().pin_memory() for x in (hq, hk, hv)] for c0, c1 in caches_rows]
    dbuf_p = [[torch.empty_like(x, device=dev) for x in p] for p in pin_p]
    dbuf_d = [[torch.empty_like(x, device=dev) for x in p] for p in pin_d]
    outs = [torch.empty(p[0].shape, dtype=tdt, device=dev) for p in pin_d]
    houts = [torch.empty(p[0].shape, dtype=tdt).pin_memory() for p in pin_d]
    O = [torch.empty(p[0].shape, dtype=tdt, device=dev) for p in pin_p]
    lse = [torch.empty(p[0].shape[:3], dtype=torch.float32, device=dev) for p in pin_p]
    colsum = [torch.empty_like(x) for x in lse]
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    side = torch.cuda.Stream(device=dev)
    back = torch.cuda.Stream(device=dev)
    last_group = {ci: max(g for g, (cj, _, _) in enumerate(groups) if cj == ci) for ci in range(nd)}

    def copy_all():
        for g, (ci, _, _) in enumerate(groups):
            for t in range(3):
                dbuf_p[g][t].copy_(pin_p[g][t], non_blocking=True)
            if g == last_group[ci]:
                for t in range(3):
                    dbuf_d[ci][t].copy_(pin_d[ci][t], non_blocking=True)

    def job(start_ev):
        side.wait_event(start_ev)
        landed = []
        with torch.cuda.stream(side):
            for g, (ci, _, _) in enumerate(groups):
                for t in range(3):
                    dbuf_p[g][t].copy_(pin_p[g][t], non_blocking=True)
                if g == last_group[ci]:
                    for t in range(3):
                        dbuf_d[ci][t].copy_(pin_d[ci][t], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(side)
                landed.append(ev)
        caches = [H2OCache(c1 - c0, w.H, w.d, w.k_heavy, w.k_local, tdt, device=dev, kv_fp8=is_kvfp8(w))
                  for c0, c1 in caches_rows]
        for c in caches:
            c.set_decode_form(args.decode_form)
        for g, (ci, b0, b1) in enumerate(groups):
            stream.wait_event(landed[g])
            c = caches[ci]
            c.prefill_rows(b0 - caches_rows[ci][0], dbuf_p[g][0], dbuf_p[g][1], dbuf_p[g][2], O=O[g], lse=lse[g],
                           colsum=colsum[g])
            if g == last_group[ci]:
                c.steps(dbuf_d[ci][0], dbuf_d[ci][1], dbuf_d[ci][2], out=outs[ci])
                done = torch.cuda.Event()
                done.record(stream)
                back.wait_event(done)
                with torch.cuda.stream(back):
                    houts[ci].copy_(outs[ci], non_blocking=True)
        stream.wait_stream(back)  # the job ends when its outputs are on the host
        return caches

    # the host link alone: every input copied once from pinned memory, nothing else running
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    copy_all()
    e1.record(stream)
    torch.cuda.synchronize()
    h2d_alone_ms = e0.elapsed_time(e1)
    n = args.steps
    nw = max(1, min(args.warmup, 3))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nw + n)]
    for i in range(nw):
        ev[i][0].record(stream)
        job(ev[i][0])
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    timed = ev[nw:]
    for a, b in timed:
        flush.zero_()
        a.record(stream)
        job(a)
        b.record(stream)
    torch.cuda.synchronize()
    ms_step, value = aggregate_over_ranks(float(np.sum([a.elapsed_time(b) for a, b in timed])), n, Bg * w.T,
                                          world, dist, dev)
    h2d = sum(x.numel() * x.element_size() for p in pin_p + pin_d for x in p)
    d2h = sum(x.numel() * x.element_size() for x in houts)
    return {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms_step,
            "pipeline": f"{ng} prompt row groups prefilled as they land into {nd} caches, each decoded once its "
                        "rows are prefilled",
            "h2d_alone": {"ms": h2d_alone_ms, "gbs": h2d / (h2d_alone_ms / 1e3) / 1e9,
                          "what": "one copy of every input buffer from pinned host memory, nothing else running"}}


# ------------------------------------------------------------ oracle timing

CPU_SAMPLE_STEPS = 65536  # decode steps of the oracle sample (the long stream's first 65,536)
CPU_SAMPLE_HEADS = 256  # at most this many heads per oracle job
CPU_SAMPLE_SECONDS = 10.0  # aim for an oracle job of about this long on the host's cores
ORACLE_S_PER_HEAD_8K = 8.5  # measured: one head's fp64 prefill at L = 8192, d = 128, one core


def sample_heads(w, cores):
    """Heads of the oracle sample: as many as keep one oracle job near
    CPU_SAMPLE_SECONDS on `cores` threads (heads run one per thread; the
    prefill cost grows as L^2 d), at least one per thread, at most
    CPU_SAMPLE_HEADS and the workload's own count."""
    per_head = ORACLE_S_PER_HEAD_8K * (w.L / 8192.0) ** 2 * (w.d / 128.0)
    per_thread = max(1, int(CPU_SAMPLE_SECONDS / max(per_head, 1e-6)))
    return max(1, min(w.nh, CPU_SAMPLE_HEADS, cores * per_thread))


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


def cpu_baseline(w, args):
    import oracle
    cores = os.cpu_count() or 1
    oracle.set_threads(cores)
    hs, T, data = oracle_sample(w, sample_heads(w, cores))
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
    hs, T, data = oracle_sample(w, sample_heads(w, cores))
    for _ in range(args.warmup):
        oracle_job(w, data)
    phases = np.array([oracle_job(w, data) for _ in range(args.steps)])
    scale = w.nh / len(hs)
    per_job = float(np.mean(phases.sum(axis=1))) * scale
    value = w.B * T / per_job
    sample = f"each step: {sample_text(w, hs, T)}"
    return {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": per_job * 1e3, "higher_is_better": True, "scaling": args.scaling,
            "vs_baseline": None, "dtype": "f64", "impl": "reference",
            "data": "synthetic: seeded per-head generator", "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": int(oracle.max_threads()),
                             "kind": "oracle", "sample": sample,
                             "phases_s": {"prefill": float(np.mean(phases[:, 0])),
                                          "decode": float(np.mean(phases[:, 1]))}},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1, help="ranks (one per GPU); started with torchrun if needed")
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG,
                    help="workload index (0 tiny, 1 OPT-6.7B-shaped, 2 OPT-30B-shaped, 3 8K prompt, 4 long stream)")
    ap.add_argument("--scaling", choices=["weak", "strong"], default="weak",
                    help="several ranks: B rows each (weak) or the B rows split over them (strong)")
    ap.add_argument("--prompt-len", type=int, default=None, help="override L (profiling captures)")
    ap.add_argument("--decode-steps", type=int, default=None, help="override T (profiling captures)")
    ap.add_argument("--decode-form", default="auto", choices=["auto", "per_step", "cooperative", "cluster", "pipelined"])
    ap.add_argument("--kv", choices=["native", "fp8"], default="native",
                    help="K/V cache storage: the workload's dtype, or e4m3 codes with a row scale (bf16 workloads)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-row-groups", type=int, default=8, help="prompt row groups copied/prefilled in turn")
    ap.add_argument("--e2e-step-groups", type=int, default=4, help="decode step groups copied/decoded in turn")
    ap.add_argument("--e2e-decode-groups", type=int, default=2,
                    help="caches of the row-pipelined end-to-end leg (each decoded once its rows are prefilled)")
    ap.add_argument("--e2e-pipeline", choices=["auto", "rows", "steps"], default="auto",
                    help="end-to-end leg: prompt row groups prefilled as they land into a few caches, each "
                         "decoded once its rows are prefilled (rows), or one cache whose decode waits for every "
                         f"row's prefill (steps); auto: rows when each cache holds at least {E2E_ROWS_MIN_HEADS} "
                         "heads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    return ap, args


def workload_of(ap, args):
    w = synth.CONFIGS[args.config]
    if args.prompt_len is not None or args.decode_steps is not None:
        L = w.L if args.prompt_len is None else args.prompt_len
        T = w.T if args.decode_steps is None else args.decode_steps
        w = w.with_(name=f"{w.name}[L={L},T={T}]", L=L, T=T)
    if args.kv == "fp8":
        if w.dtype != "bf16":
            ap.error("--kv fp8 needs a bf16 workload")
        w = w.with_(name=w.name + FP8_SUFFIX)
    return w


def main():
    ap, args = parse_args()
    w = workload_of(ap, args)
    env_world = os.environ.get("WORLD_SIZE")
    if env_world is None and args.gpus > 1 and args.impl == "ours":
        sys.exit(relaunch_under_torchrun(args.gpus))
    rank = int(os.environ.get("RANK", "0"))
    world = int(env_world or "1")
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if env_world is not None and args.gpus != world and args.gpus != 1:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}")
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

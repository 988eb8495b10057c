"""The bench's host-side legs on CPU: the oracle baseline and the reference
arm (both time the fp64 oracle on a bounded sample of the workload) and the
JSON line the reference arm prints."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import bench
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_cpu_baseline_times_the_whole_small_job():
    cb = bench.cpu_baseline(synth.TINY, None)
    assert cb["kind"] == "oracle" and cb["unit"] == "tokens/s"
    assert cb["value"] > 0 and cb["cores"] >= 1
    assert cb["phases_s"]["prefill"] > 0 and cb["phases_s"]["decode"] > 0
    assert "(the full job)" in cb["sample"]


def test_oracle_sample_is_bounded_to_the_first_decode_steps():
    w = synth.LONG_STREAM.with_(name="stream_sample", B=1, H=1, L=16, k_heavy=8, k_local=8,
                                T=bench.CPU_SAMPLE_STEPS + 100)
    hs, T, data = bench.oracle_sample(w, bench.CPU_SAMPLE_HEADS)
    assert hs == [0] and T == bench.CPU_SAMPLE_STEPS
    q = data[3]
    assert q.shape[0] == bench.CPU_SAMPLE_STEPS
    assert f"the first {T} of {w.T} decode steps" in bench.sample_text(w, hs, T)


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "0",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 3 and line["warmup"] == 3
    assert line["value"] > 0 and line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["value"] == line["value"] and line["cpu_baseline"]["kind"] == "oracle"
    assert set(line["cpu_baseline"]["phases_s"]) == {"prefill", "decode"}
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == synth.TINY.name


def test_default_workload_is_the_largest_single_gpu_one():
    """The bench line is quoted on the 8K-prompt shape: the largest K/V cache
    and the most prefill work of the single-GPU workloads."""
    w = synth.CONFIGS[bench.DEFAULT_CONFIG]
    assert w is synth.PREFILL_HEAVY
    single = [c for c in synth.CONFIGS if not bench.streamed(c)]
    assert bench.kv_read_bytes(w) == max(bench.kv_read_bytes(c) for c in single)
    assert bench.score_pass_flops(w) == max(bench.score_pass_flops(c) for c in single)
    assert bench.kv_read_bytes(w) > bench.L2_RESIDENT_BYTES  # read from HBM every step


def test_oracle_sample_heads_are_bounded():
    cores = 16
    assert bench.sample_heads(synth.PREFILL_HEAVY, cores) == cores  # one 8K-prompt head per thread
    assert bench.sample_heads(synth.OPT_6_7B, cores) == synth.OPT_6_7B.nh  # the whole job
    assert bench.sample_heads(synth.TINY, cores) == synth.TINY.nh
    assert bench.sample_heads(synth.OPT_30B, cores) == bench.CPU_SAMPLE_HEADS

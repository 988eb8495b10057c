"""The stored ncu DRAM-traffic records (profiles/traffic.json) that the bench
line quotes as `roofline.traffic`.  Each record names the kernel's source
file and the hash of the source it was captured from, and the bench drops a
record whose source has changed since.  These checks keep the committed
records in step with the committed kernels and check the bench's lookup."""
from __future__ import annotations

import hashlib
import json
import os

import pytest

import bench
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
RECORDS = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
# the bench names a run with an fp8 K/V cache by its workload plus a suffix
WORKLOADS = {w.name: w for w in synth.CONFIGS}
WORKLOADS.update({w.name + bench.FP8_SUFFIX: w.with_(name=w.name + bench.FP8_SUFFIX) for w in synth.CONFIGS})


@pytest.mark.parametrize("key", sorted(RECORDS))
def test_record_matches_the_committed_source(key):
    rec = RECORDS[key]
    kernel, workload = key.split("@", 1)
    assert workload in WORKLOADS, workload
    src = os.path.join(ROOT, rec["source"])
    assert os.path.exists(src), rec["source"]
    assert kernel in open(src).read(), f"{kernel} is not defined in {rec['source']}"
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    assert rec["source_sha"] == sha, f"{rec['source']} changed since this capture: take it again, or remove the record"
    assert rec["dram_bytes_per_launch"] > 0
    assert os.path.exists(os.path.join(ROOT, rec["profile"])), rec["profile"]


@pytest.mark.parametrize("key", sorted(RECORDS))
def test_bench_quotes_the_record(key):
    kernel, workload = key.split("@", 1)
    value, where = bench.traffic_for(kernel, WORKLOADS[workload])
    assert value == RECORDS[key]["dram_bytes_per_launch"]
    assert RECORDS[key]["source_sha"] in where


def test_bench_drops_a_record_of_another_source(tmp_path, monkeypatch):
    key = sorted(RECORDS)[0]
    kernel, workload = key.split("@", 1)
    stale = dict(RECORDS)
    stale[key] = dict(RECORDS[key], source_sha="0" * 16)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(stale))
    src = tmp_path / RECORDS[key]["source"]
    src.parent.mkdir(parents=True)
    src.write_bytes(open(os.path.join(ROOT, RECORDS[key]["source"]), "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    value, why = bench.traffic_for(kernel, WORKLOADS[workload])
    assert value is None and "changed since the stored capture" in why

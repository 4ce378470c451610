"""Host logic of bench.py that needs no GPU: which DRAM-traffic record a bench
line may quote, and the kernel each configuration is keyed by.

A record (profiles/dram_traffic.json) holds the dram bytes of one kernel
launch measured by ncu on one workload; the bench quotes it only for that
workload and only while the kernel's sources hash to the recorded value.
"""
import argparse
import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from attention_blackwell_gb300 import workloads as W  # noqa: E402


def _args(**kw):
    a = dict(deterministic=False, bwd_kernel=0, exp2_emu=0, fwd_kernel=2)
    a.update(kw)
    return argparse.Namespace(**a)


@pytest.fixture
def fake_root(tmp_path, monkeypatch):
    """A tree with one kernel source and one traffic record over it."""
    (tmp_path / "profiles").mkdir()
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    rec = {"fwd_x": {"sources": ["k.cu"], "sources_sha": sha, "dram_bytes_per_launch": 12345,
                     "workload": "large: B=4 ...", "from": "profiles/x.md"}}
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def test_traffic_quoted_for_its_own_workload_only(fake_root):
    assert bench.kernel_traffic("fwd_x", "large") == 12345
    assert bench.kernel_traffic("fwd_x", "causal") is None      # counters taken on another workload
    assert bench.kernel_traffic("fwd_y", "large") is None       # no record


def test_traffic_dropped_once_the_sources_change(fake_root):
    (fake_root / "k.cu").write_text("kernel v2\n")
    assert bench.kernel_traffic("fwd_x", "large") is None


def test_traffic_key_follows_the_kernel_that_runs():
    large, varlen = W.WORKLOADS["large"], W.WORKLOADS["varlen"]
    assert bench.traffic_key(_args(), large, "fwd") == "fwd_pair"
    assert bench.traffic_key(_args(fwd_kernel=0), large, "fwd") == "fwd_pingpong"
    assert bench.traffic_key(_args(exp2_emu=1), large, "fwd") == "fwd_pair"
    assert bench.traffic_key(_args(), varlen, "fwd") == "fwd_pair"
    assert bench.traffic_key(_args(), large, "bwd") == "bwd"
    assert bench.traffic_key(_args(bwd_kernel=1), large, "bwd") == "bwd_pair"
    assert bench.traffic_key(_args(bwd_kernel=1, deterministic=True), large, "bwd") == "bwd_pair"
    assert bench.traffic_key(_args(bwd_kernel=1), varlen, "bwd") == "bwd_pair"
    assert bench.traffic_key(_args(), W.WORKLOADS["large_d256"], "fwd") == "fwd_d256"
    assert bench.traffic_key(_args(), W.WORKLOADS["large_d64"], "bwd") == "bwd_d64"


def test_committed_records_name_existing_workloads_and_sources():
    recs = json.load(open(os.path.join(ROOT, "profiles", "dram_traffic.json")))
    for name, rec in recs.items():
        assert rec["workload"].split(":")[0] in W.WORKLOADS, name
        for src in rec["sources"]:
            assert os.path.exists(os.path.join(ROOT, src)), (name, src)
        assert rec["dram_bytes_per_launch"] > 0

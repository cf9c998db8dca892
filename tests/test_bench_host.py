"""Host logic of the bench's roofline fields (CPU): the peak comes from the
measured file, and the DRAM traffic figure is given only while the
chain kernel's sources are the ones the committed ncu summary was taken on."""
import json
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_peak_is_the_measured_copy_bandwidth():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(p):
        assert bench.peaks() == (6800.0, "fallback")
        return
    assert bench.peaks() == (float(json.load(open(p))["hbm_gbs"]), "measured")


def _profile_fields():
    p = os.path.join(ROOT, "profiles", "gemm_tc_kernel.llama7b_shapes.md")
    fields = {}
    for line in open(p):
        if ":" in line and line.split(":")[0] in ("traffic_over_algorithmic", "gemm_sources_sha256"):
            k, v = line.split(":", 1)
            fields[k] = v.strip()
    return fields


def test_traffic_only_for_the_profiled_sources(monkeypatch):
    f = _profile_fields()
    assert len(f["gemm_sources_sha256"]) == 64 and 0.9 < float(f["traffic_over_algorithmic"]) < 1.5
    monkeypatch.setattr(bench, "gemm_source_sha256", lambda: f["gemm_sources_sha256"])
    assert bench.gemm_traffic_per_launch(4.0e8) == pytest.approx(float(f["traffic_over_algorithmic"]) * 4.0e8)
    monkeypatch.setattr(bench, "gemm_source_sha256", lambda: "0" * 64)
    assert bench.gemm_traffic_per_launch(4.0e8) is None


def test_source_hash_covers_the_chain_kernel_files():
    names = set(bench.GEMM_SOURCES)
    assert {"gemm.cu", "attn_phase.cuh", "model.cuh"} <= names
    for n in names:
        assert os.path.exists(os.path.join(ROOT, "speculative_decoding_verify_04_gb300", "csrc", n))
    assert len(bench.gemm_source_sha256()) == 64

"""Host-side pieces of bench.py that decide what the reported numbers mean:
the frozen algorithmic-work formulas and the staleness check of the
committed DRAM-traffic record (CPU only)."""

import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


@pytest.mark.parametrize("K,V,fwd", [(64, 64, 46.4e3), (64, 128, 79.2e3), (128, 128, 140.6e3), (128, 256, 255.3e3)])
def test_forward_flops_per_token_head(K, V, fwd):
    # 6KV (the recurrence) + gram C^2 K + inverse C^3/3 + w C^2 K + u C^2 V
    # + Q K^T C^2 K + P Delta C^2 V, per token (C = 64)
    assert bench.fwd_flops(K, V) == pytest.approx(fwd, rel=1e-3)


def test_bytes_and_backward_per_token_head():
    assert bench.fwd_bytes(128, 128) == 1030          # q, k, v, o bf16; g fp32; beta bf16
    assert bench.bwd_bytes(128, 256) == 2572          # + dO in; dq, dk, dv, dg, dbeta out
    assert bench.bwd_flops(128, 256) == pytest.approx(700e3, rel=2e-3)


def test_target_workload_totals():
    """B=4, H=16, T=4096, d_k=d_v=128: 36.9 GFLOP and 274.2 MB (with the 4 MiB
    final state), a roofline time of ~40 us on ~6.8 TB/s."""
    th, f, b, fb, bb = bench.workload_totals(4, 4096, 16, 128, 128)
    assert th == 4 * 4096 * 16
    assert f == pytest.approx(36.9e9, rel=1e-3)
    assert b == 1030 * th + 4 * 128 * 128 * 64 == 274_202_624
    assert fb > 2 * f and bb > b


def test_traffic_record_only_counts_for_its_sources(tmp_path, monkeypatch):
    csrc = tmp_path / "linear_attention_sequence_chunked_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = csrc / "kernel.cu"
    src.write_text("// kernel v1\n")
    rec = {"sources": {"kernel.cu": hashlib.sha256(src.read_bytes()).hexdigest()}, "bytes_per_launch": 123}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic() == 123
    src.write_text("// kernel v2\n")                     # the kernel changed since the capture
    assert bench.load_traffic() is None
    rec["sources"] = {}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.load_traffic() is None                  # a record naming no sources counts for nothing


def test_committed_traffic_record_matches_the_tree():
    """The committed record, if it claims a value, was taken on these sources."""
    v = bench.load_traffic()
    assert v is None or v > bench.workload_totals(4, 4096, 16, 128, 128)[2]

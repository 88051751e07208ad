"""Host logic of bench.py that needs no GPU: the roofline's traffic figure is
taken from the recorded ncu capture only while it describes the current kernel
sources and the same GEMM sequence; the fused-conv pass has no conv-gate GEMMs."""

import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402
from block_diffusion_drafter_inject_gb300.build import source_fingerprint  # noqa: E402


@pytest.fixture
def record(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))

    def write(**kw):
        rec = dict(launches_per_pass=21, dram_bytes_per_pass=123456789,
                   source_fingerprint=source_fingerprint())
        rec.update(kw)
        (prof / "gemm_roofline_traffic.json").write_text(json.dumps(rec))
    return write


def test_traffic_reported_for_matching_sources(record):
    record()
    assert bench.stored_traffic(21) == 123456789


def test_traffic_null_once_sources_change(record):
    record(source_fingerprint="0" * 64)
    assert bench.stored_traffic(21) is None


def test_traffic_null_for_another_sequence(record):
    record()
    assert bench.stored_traffic(25) is None


def test_traffic_null_without_record(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.stored_traffic(21) is None


def test_fingerprint_is_machine_independent_and_tracks_sources():
    from block_diffusion_drafter_inject_gb300 import build
    fp = source_fingerprint()
    assert len(fp) == 64 and fp == source_fingerprint()
    assert build._fingerprint().startswith(fp + "|")


def test_pass_gemms_fused_conv_has_no_gate_gemms():
    cfg = synth.preset("full")
    b1 = bench.pass_gemms(cfg, 1, 8)
    assert len(b1) == 5 * 4 + 1  # QKV, O, gate/up, down per layer + lm_head
    assert not any(".conv_w." in g[3] for g in b1)
    b32 = bench.pass_gemms(cfg, 32, 8)
    assert sum(".conv_w." in g[3] for g in b32) == 5 * 4

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


def _copy_sources(dst):
    """The library sources and headers of this checkout copied under `dst`."""
    import shutil
    from block_diffusion_drafter_inject_gb300 import build
    for d in (build.CSRC, build.INCLUDE):
        rel = os.path.relpath(d, build.ROOT)
        shutil.copytree(d, os.path.join(dst, rel),
                        ignore=shutil.ignore_patterns("__pycache__"))


def test_fingerprint_is_the_same_in_another_checkout_path(tmp_path):
    a, b = tmp_path / "one", tmp_path / "somewhere" / "else" / "two"
    _copy_sources(str(a))
    _copy_sources(str(b))
    fa, fb = source_fingerprint(str(a)), source_fingerprint(str(b))
    assert fa == fb == source_fingerprint()
    # ... and still follows the sources
    hdr = b / "include" / "dflash.h"
    hdr.write_text(hdr.read_text() + "\n/* changed */\n")
    assert source_fingerprint(str(b)) != fa


def test_portable_flags_make_checkout_paths_relative():
    from block_diffusion_drafter_inject_gb300 import build
    flags = ["-O3", "-I", "/x/y/repo/include", "-I", "/x/y/repo/pkg/csrc", "-I", "/opt/other"]
    assert build.portable_flags(flags, "/x/y/repo") == [
        "-O3", "-I", "include", "-I", os.path.join("pkg", "csrc"), "-I", "/opt/other"]


def test_bench_replicas_reach_world_two_on_cpu():
    """`bench.py --gpus 2` with no WORLD_SIZE launches two ranks itself; the CPU
    self-check of the replica plumbing (gloo) sees world 2 and the max over ranks."""
    import subprocess
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2",
                        "--replica-selftest"], capture_output=True, text=True, timeout=300,
                       env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = [l for l in r.stdout.splitlines() if l.startswith("{")][-1]
    out = json.loads(line)
    assert out["world"] == 2 and out["max_step"] == 2.0 and out["value"] == 1000.0


def test_pass_gemms_fused_conv_has_no_gate_gemms():
    cfg = synth.preset("full")
    b1 = bench.pass_gemms(cfg, 1, 8)
    assert len(b1) == 5 * 4 + 1  # QKV, O, gate/up, down per layer + lm_head
    assert not any(".conv_w." in g[3] for g in b1)
    b32 = bench.pass_gemms(cfg, 32, 8)
    assert sum(".conv_w." in g[3] for g in b32) == 5 * 4

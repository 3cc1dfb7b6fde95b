"""bench.py's host-side bookkeeping, on the CPU: the projection-source digest
that keys the recorded ncu traffic (code only, the projection's part of the
shared header), the traffic lookup by workload and plan, and the L2 flush
description carried in the JSON line."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_drops_comments_blank_lines_and_indentation():
    src = b"int a;  // the count\n\n    // a whole-line comment\n  int b = 2; //\n"
    assert bench._code_only(src) == b"int a;\nint b = 2;"
    assert bench._code_only(b"// only a comment\n") == b""


def test_projection_part_keeps_header_and_projection_section():
    text = (b"#pragma once\nshared;\n// ---- rows: gather\ngather_only;\n// ---- projection (a4)\nproj;\n"
            b"// ---- gate and residual\ngate_only;\n")
    part = bench._projection_part(text)
    assert b"shared;" in part and b"proj;" in part
    assert b"gather_only" not in part and b"gate_only" not in part
    # without the section markers the whole text counts
    assert bench._projection_part(b"no markers here") == b"no markers here"


def test_digest_covers_the_projection_sources():
    d = bench.source_digest(bench.GEMM_SOURCES)
    assert len(d) == 16 and int(d, 16) >= 0
    assert d == bench.source_digest(bench.GEMM_SOURCES)       # deterministic


def test_recorded_traffic_matches_workload_digest_and_plan(tmp_path, monkeypatch):
    digest = bench.source_digest(bench.GEMM_SOURCES)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "wkv_gemm_traffic.txt").write_text(
        "# comment line\n"
        f"workload=w1 kernel=k plan=1x100 source_sha256={digest} dram_bytes_per_launch=123 read=120 write=3\n"
        f"workload=w4 kernel=k plan=1x152pr16x4 source_sha256={digest} dram_bytes_per_launch=7 read=5 write=2\n"
        f"workload=w2 kernel=k source_sha256=0000000000000000 dram_bytes_per_launch=456 read=450 write=6\n"
        f"workload=w3 kernel=k source_sha256={digest} dram_bytes_per_launch=789 read=780 write=9\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_digest", lambda files: digest)
    one = bench.plan_key(dict(splits=1, ctas=100, cta_pairs=0, rem_tiles=0, rem_splits=0))
    assert one == "1x100"
    assert bench.recorded_traffic("w1", one) == 123.0
    assert bench.recorded_traffic("w1") == 123.0                 # no plan given: the record stands
    assert bench.recorded_traffic("w1", "3x152") is None          # captured with another plan
    assert bench.recorded_traffic("w2", one) is None              # captured on other source
    assert bench.recorded_traffic("w3", "8x152") == 789.0         # the record names no plan
    assert bench.recorded_traffic("absent", one) is None
    pairs = bench.plan_key(dict(splits=1, ctas=152, cta_pairs=1, rem_tiles=16, rem_splits=4))
    assert pairs == "1x152pr16x4" and bench.recorded_traffic("w4", pairs) == 7.0
    assert bench.recorded_traffic("w4", "1x152p") is None         # pairs without the remainder split
    fused = bench.plan_key(dict(splits=1, ctas=152, cta_pairs=1, rem_tiles=0, rem_splits=0, fused_gate=1))
    assert fused == "1x152pf" and bench.recorded_traffic("w4", fused) is None


def test_committed_traffic_records_add_up():
    """Each committed record's total is its reads plus its writes, and it names
    the kernel, the plan and the source digest it was captured on (a record
    for an older source is simply not reported)."""
    lines = [l for l in open(os.path.join(ROOT, "profiles", "wkv_gemm_traffic.txt")) if l.startswith("workload=")]
    assert lines
    for l in lines:
        kv = dict(t.split("=", 1) for t in l.split() if "=" in t)
        assert float(kv["dram_bytes_per_launch"]) == float(kv["read"]) + float(kv["write"])
        assert len(kv["source_sha256"]) == 16 and "kernel" in kv and "plan" in kv


def test_l2_flush_description_names_write_and_read():
    assert "write" in bench.L2_NOTE and "read" in bench.L2_NOTE

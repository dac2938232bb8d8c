"""The host side of bench.py on the CPU: clock-sample summaries, the traffic-table
gate, the roofline arithmetic, and the reference arm's JSON line."""
import json
import os
import subprocess
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _line(t, sm, mx, reasons=("Not Active",) * 4):
    return (t, f"0, {sm}, {mx}, 900.5, 0x0, " + ", ".join(reasons))


def test_clock_summary_median_window_and_reasons():
    s = bench.ClockSampler(0)
    t0 = 1000.0
    s.lines = [_line(t0 - 1, 100, 2070), _line(t0 + 0.1, 2070, 2070), _line(t0 + 0.2, 1900, 2070),
               _line(t0 + 0.3, 2070, 2070, ("Not Active", "Not Active", "Not Active", "Active")),
               _line(t0 + 5, 50, 2070, ("Active",) * 4)]
    out = s.summary(t0, t0 + 1)
    assert out["samples"] == 3 and out["sm_mhz"] == 2070 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]           # samples outside the window are ignored
    empty = s.summary(t0 + 10, t0 + 11)
    assert empty["samples"] == 0 and empty["sm_mhz"] is None


def test_traffic_table_follows_the_kernel_sources(tmp_path, monkeypatch):
    """A kernel's DRAM bytes count only while its own sources are unchanged since the capture."""
    prof = tmp_path / "profiles"
    prof.mkdir()
    csrc = tmp_path / "top_kl_distill_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in set(bench.ROW_SOURCES) | set(bench.TOPK_SOURCES):
        (csrc / f).write_text(f"// {f}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    row_hash = bench.sources_hash(bench.ROW_SOURCES)
    (prof / "ncu_traffic.json").write_text(json.dumps(
        {"kernels": {"ce_fused": {"dram_bytes_per_launch": 123, "sources_sha256": row_hash},
                     "topk_k256": {"dram_bytes_per_launch": 456, "sources_sha256": "0" * 64}}}))
    assert bench.kernel_traffic("ce_fused") == 123
    assert bench.kernel_traffic("topk_k256") is None           # captured from other sources
    assert bench.kernel_traffic("no_such_kernel") is None
    (csrc / "rows.cu").write_text("// changed\n")               # the row kernels changed since the capture
    assert bench.kernel_traffic("ce_fused") is None


def test_sources_hash_is_stable_and_source_sensitive():
    assert bench.sources_hash(bench.ROW_SOURCES) == bench.sources_hash(bench.ROW_SOURCES)
    assert len(bench.sources_hash(bench.ROW_SOURCES)) == 64
    assert bench.sources_hash(bench.ROW_SOURCES) != bench.sources_hash(bench.TOPK_SOURCES)


def test_roofline_arithmetic():
    class C:
        def kernel_bytes(self):
            return 131_078_144

    r = bench.roofline(C(), 0.0282, 6783.8, "measured", "ce_fused_test")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - 131_078_144 / 28.2e-6 / 1e9) < 0.1
    assert abs(r["frac"] - r["achieved"] / 6783.8) < 1e-4
    assert r["traffic"] is None


def test_reference_arm_prints_one_json_line():
    t0 = time.time()
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                          "--warmup", "3"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "cpu_baseline", "e2e", "config"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    assert time.time() - t0 < 300

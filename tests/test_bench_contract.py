"""The benchmark's JSON line and its host-side pieces, checked on the CPU.

bench.py's reference arm runs the float64 oracle on the host, so its full
output line can be produced and validated here; the clock-sample summary is
checked on synthetic nvidia-smi lines.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

REQUIRED = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
            "vs_baseline", "dtype", "data", "config")


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                          "--warmup", "1", "--workload", "single_head_T256_d64"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    for k in REQUIRED:
        assert k in d, k
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 1 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "single_head_T256_d64"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_clock_summary_windows():
    c = bench.ClockSampler(0)
    c.lines = [(1.00, "0, 2070, 2070, 900, 0x0, Not Active, Not Active, Not Active, Not Active"),
               (1.05, "0, 2070, 2070, 950, 0x4, Not Active, Not Active, Not Active, Active"),
               (1.10, "0, 2055, 2070, 1000, 0x0, Not Active, Not Active, Not Active, Not Active")]
    inside = c.summary(1.04, 1.11)
    assert inside["window"] == "timed region" and inside["samples"] == 2 and inside["sm_mhz"] == 2062.5
    assert inside["reasons"] == ["sw_power_cap"]
    short = c.summary(1.01, 1.04)  # no sample inside: the two around it
    assert short["samples"] == 2 and "before and after" in short["window"]
    none = bench.ClockSampler(0).summary(0.0, 1.0)
    assert none["reasons"] == ["unsampled"] and none["sm_mhz"] is None


def test_measured_traffic_is_tied_to_the_source():
    # a recorded figure is reported only while the kernel source it was taken on is unchanged
    for w in bench.NCU_TRAFFIC:
        v = bench.measured_traffic(w)
        assert v is None or v == bench.NCU_TRAFFIC[w]["bytes"]
    assert bench.measured_traffic("no_such_workload") is None


def test_peaks_fall_back_when_unmeasured(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.load_peaks()
    assert p["source"] == "fallback" and p["bf16_tflops"] == 1900.0

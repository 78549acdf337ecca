"""bench.py on the CPU: the reference arm's JSON line (the oracle timed on a
bounded sample), the gating of the recorded DRAM traffic by the kernel-source
hash, and the command line."""
import json
import os
import subprocess
import sys

import pytest

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_reference_arm_prints_one_line_with_the_same_metric():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "square_512", "--steps", "2", "--warmup", "0"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["value"] > 0
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["config"]["name"] == "square_512" and d["gpu_launches"] == 0


def test_recorded_traffic_is_gated_by_the_kernel_source_hash(monkeypatch):
    key = ("square_16384x16384x4096", "grouped", True)
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)["square_16384x16384x4096|grouped|cross=on"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: rec["kernel_source_sha256"])
    assert bench.recorded_traffic(*key) == rec["dram_bytes_per_launch"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 64)
    assert bench.recorded_traffic(*key) is None
    assert bench.recorded_traffic("no_such_workload", "grouped", True) is None


def test_kernel_source_hash_covers_the_kernel_sources():
    h = bench.kernel_source_hash()
    assert len(h) == 64 and int(h, 16) >= 0


@pytest.mark.parametrize("sweep", ["order", "ksweep", "kernel", "persistence", "cublas", "splitk",
                                   "outdtype", "ragged", "schedule", "tail"])
def test_sweeps_parse(sweep):
    a = bench.parse_args(["--sweep", sweep, "--steps", "3", "--warmup", "3"])
    assert a.sweep == sweep and a.steps == 3 and a.warmup == 3


def test_defaults_finish_within_minutes():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and 1 <= a.steps <= 1000


def test_roofline_peak_follows_the_observed_regime():
    peaks = {"bf16_tflops": 1914.3, "bf16_tflops_sustained": 1748.8}
    unthrottled = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    peak, note = bench.roofline_peak(peaks, "measured", unthrottled)
    assert peak == 1914.3 and "burst" in note
    capped = {"sm_mhz": 1400.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    peak, note = bench.roofline_peak(peaks, "measured", capped)
    assert peak == 1748.8 and "sustained" in note and "sw_power_cap" in note
    low = {"sm_mhz": 1500.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert bench.roofline_peak(peaks, "measured", low)[0] == 1748.8
    # without a sustained figure, or without clock samples: the burst peak
    assert bench.roofline_peak({"bf16_tflops": 1914.3}, "measured", capped)[0] == 1914.3
    assert bench.roofline_peak(peaks, "measured", None)[0] == 1914.3


def test_target_is_stated_on_one_P():
    t = bench.target_line(1777.0, 2500.0)
    assert t["P_tflops"] == 2500.0 and t["goal_frac"] == 0.70
    assert abs(t["frac_of_P"] - 1777.0 / 2500.0) < 1e-12 and t["met"] is True
    assert bench.target_line(1737.7, 2500.0)["met"] is False

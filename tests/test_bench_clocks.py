"""bench.py's clock sampler: live before the timed region opens, and keeping
only the samples that arrive inside the window it is given (a fake
nvidia-smi on PATH stands in for the real one)."""
import os
import stat
import time

import pytest

from tests.conftest import ROOT  # noqa: F401  (puts the repo root on sys.path)

FAKE = """#!/usr/bin/env python3
import sys, time
period = 0.05
for a in sys.argv[1:]:
    if a.startswith("-lms="):
        period = int(a[5:]) / 1000.0
time.sleep(0.3)  # slow start, like the real tool
i = 0
while True:
    cap = "Active" if i % 2 else "Not Active"
    print(f"0, {1900 + i}, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, {cap}", flush=True)
    i += 1
    time.sleep(period)
"""


@pytest.fixture
def fake_smi(tmp_path, monkeypatch):
    exe = tmp_path / "nvidia-smi"
    exe.write_text(FAKE)
    exe.chmod(exe.stat().st_mode | stat.S_IXUSR)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    return exe


def test_sampler_is_live_on_entry_and_keeps_its_window(fake_smi):
    import bench
    with bench.ClockSampler(0, period_ms=20) as clk:
        assert clk.rows, "entering waits for the first sample"
        t0 = time.perf_counter()
        time.sleep(0.3)
        t1 = time.perf_counter()
        time.sleep(0.2)
        clk.set_window(t0, t1, "timed region")
        inside = clk.count(t0, t1)
    s = clk.summary()
    assert s["samples"] == inside >= 5
    assert s["samples"] < len(clk.rows)
    assert s["sm_max_mhz"] == 2070.0
    assert 1900 <= s["sm_mhz"] < 1900 + len(clk.rows)
    assert s["reasons"] == ["sw_power_cap"]
    assert s["window"] == "timed region"


def test_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    import bench
    monkeypatch.setenv("PATH", str(tmp_path))
    with bench.ClockSampler(0) as clk:
        pass
    s = clk.summary()
    assert s["reasons"] == ["unavailable"] and s["samples"] == 0


def test_peak_is_burst_unless_a_seconds_long_region_ran_under_the_cap():
    """The roofline denominator: the burst bf16 figure, unless the timed
    region lasted seconds (as the sustained figure's own measurement did) and
    ran under the power cap; FP8 and FP4 scale it by the nominal dense ratios
    2 and 6."""
    import bench
    peaks = {"bf16_tflops": 1971.4, "bf16_tflops_sustained": 1745.6}
    assert bench.peak_tflops(peaks, "fp8", False)[0] == 2 * 1971.4
    assert bench.peak_tflops(peaks, "fp8", True)[0] == 2 * 1745.6
    assert bench.peak_tflops(peaks, "fp4", False)[0] == 6 * 1971.4
    assert bench.peak_tflops(peaks, "int8", True)[0] == 1745.6
    assert "bf16_tflops_sustained" in bench.peak_tflops(peaks, "fp8", True)[1]
    capped = {"reasons": ["sw_power_cap"]}
    assert bench.use_sustained_peak(capped, 3.0)
    assert not bench.use_sustained_peak(capped, 0.58)  # a sub-second region is a burst
    assert not bench.use_sustained_peak({"reasons": []}, 3.0)
    assert not bench.use_sustained_peak({"reasons": ["unavailable"]}, 3.0)


def test_summary_of_a_sub_window(fake_smi):
    """summary(window) keeps the samples of that window only (the peak choice
    reads the timed region alone, not the untimed steps after it)."""
    import bench
    with bench.ClockSampler(0, period_ms=20) as clk:
        t0 = time.perf_counter()
        time.sleep(0.25)
        t1 = time.perf_counter()
        time.sleep(0.25)
        t2 = time.perf_counter()
        clk.set_window(t0, t2, "timed region and the untimed steps after it")
    whole, part = clk.summary(), clk.summary((t0, t1))
    assert 0 < part["samples"] < whole["samples"]
    assert clk.summary((t2 + 10, t2 + 20))["samples"] == 0

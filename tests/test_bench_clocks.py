"""bench.py's reading of the nvidia-smi samples taken during the timed region: the median
SM clock under load, the maximum clock, and every throttle reason seen active (a run that
saw a hardware or thermal slowdown is not a valid measurement)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _sampler(tmp_path, lines):
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    s.proc = object()  # as if nvidia-smi had been started
    return s


def test_median_max_and_no_reasons(tmp_path):
    # index, sm MHz, max MHz, power, active mask, hw, hw thermal, sw thermal, sw power cap
    lines = ["0, 2032, 2032, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 1980, 2032, 950.3, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 2010, 2032, 940.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    out = _sampler(tmp_path, lines).summary()
    assert out["sm_mhz"] == 2010.0 and out["sm_max_mhz"] == 2032.0
    assert out["reasons"] == [] and out["samples"] == 3


def test_active_reasons_are_reported_and_bad_lines_skipped(tmp_path):
    lines = ["0, 2032, 2032, 1090.0, 0x4, Not Active, Not Active, Not Active, Active",
             "garbage line",
             "0, [N/A], 2032, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 1800, 2032, 1100.0, 0x40, Not Active, Active, Not Active, Not Active"]
    out = _sampler(tmp_path, lines).summary()
    assert out["samples"] == 2
    assert out["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert out["sm_mhz"] == 1916.0


def test_without_nvidia_smi(tmp_path):
    s = bench.ClockSampler(0)
    s.proc = None
    out = s.summary()
    assert out["sm_mhz"] is None and out["reasons"] == ["nvidia-smi unavailable"]

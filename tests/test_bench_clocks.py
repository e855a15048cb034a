"""bench.py's clock summary on CPU, from synthetic nvidia-smi lines (no GPU).

The bench samples clocks every 20 ms around a timed region and must report
only the samples taken while the timed calls ran, with their throttle
reasons, falling back to the samples around the region (and saying so) only
when none fell inside it.
"""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _line(sm, power=900.0, cap="Not Active", thermal="Not Active"):
    return f"0, {sm}, 2070, {power}, 0x0000000000000004, Not Active, {thermal}, Not Active, {cap}"


def _sampler(lines, windows):
    s = bench.ClockSampler(0)
    s.lines = lines
    s.windows = windows
    return s


def test_only_samples_inside_the_timed_calls():
    lines = [(0.00, _line(2070)), (0.02, _line(2070)),           # before: idle, full clock
             (1.00, _line(1600, cap="Active")), (1.02, _line(1620, cap="Active")),
             (1.04, _line(1640, cap="Active")),                     # inside the window
             (2.00, _line(2070))]                                   # after
    out = _sampler(lines, [(0.99, 1.03)]).summary()
    assert out["samples"] == 3 and out["samples_total"] == 6
    assert out["sm_mhz"] == 1620 and out["sm_mhz_min"] == 1600
    assert out["reasons"] == ["sw_power_cap"]
    assert out["basis"].startswith("samples taken during")


def test_several_windows_and_reasons():
    lines = [(0.5, _line(2000, thermal="Active")), (1.5, _line(1900)), (3.0, _line(1000, cap="Active"))]
    out = _sampler(lines, [(0.4, 0.6), (1.4, 1.6)]).summary()
    assert out["samples"] == 2 and out["sm_mhz"] == 1950
    assert out["reasons"] == ["hw_thermal_slowdown"]


def test_fallback_when_no_sample_falls_inside():
    lines = [(0.0, _line(2070)), (0.5, _line(2050))]
    out = _sampler(lines, [(0.2, 0.21)]).summary()
    assert out["samples"] == 2
    assert out["basis"].startswith("no sample fell inside")


def test_no_samples_at_all():
    out = _sampler([], [(0.0, 1.0)]).summary()
    assert out["sm_mhz"] is None and out["samples"] == 0


def test_timed_region_marks_the_active_sampler():
    import torch
    s = bench.ClockSampler(0)
    bench.ClockSampler.active = s
    try:
        bench.timed_region(lambda i: None, 3, 1, torch.device("cpu"), lambda: None)
    finally:
        bench.ClockSampler.active = None
    assert len(s.windows) == 1 and s.windows[0][1] >= s.windows[0][0]

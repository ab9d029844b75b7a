"""Host logic of bench.py's clock sampling: only samples inside the timed
window count, and the throttle reasons of those samples are reported."""
import datetime

import bench


def _line(t, sm, reasons=("Not Active",) * 4):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return ", ".join([ts, "0", str(sm), "2070", "900.0", "0x0"] + list(reasons)) + "\n"


def test_samples_outside_the_window_are_dropped():
    s = bench.ClockSampler(0)
    t0 = 1_700_000_000.0
    s.lines = [_line(t0 - 1.0, 1200), _line(t0 + 0.010, 2070), _line(t0 + 0.030, 2070),
               _line(t0 + 2.0, 1200, ("Not Active", "Active", "Not Active", "Not Active"))]
    c = s.summary(t0, t0 + 0.040)
    assert c["samples"] == 2
    assert c["sm_mhz"] == 2070 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == []


def test_throttle_reasons_inside_the_window_are_reported():
    s = bench.ClockSampler(0)
    t0 = 1_700_000_000.0
    s.lines = [_line(t0 + 0.01, 1800, ("Not Active", "Not Active", "Not Active", "Active"))]
    c = s.summary(t0, t0 + 0.02)
    assert c["samples"] == 1 and c["reasons"] == ["sw_power_cap"]


def test_a_window_shorter_than_the_period_takes_the_nearest_sample():
    s = bench.ClockSampler(0)
    t0 = 1_700_000_000.0
    s.lines = [_line(t0 - 0.5, 1500), _line(t0 + 0.03, 2070)]
    c = s.summary(t0, t0 + 0.01)
    assert c["samples"] == 0 and c["sm_mhz"] == 2070


def test_nvml_samples_are_summarised_like_smi_lines():
    """In-process NVML samples (time, SM MHz, max MHz, reason bits): the same window cut and
    reason names; the power-cap bit alone is reported, not rejected."""
    s = bench.NvmlClockSampler(0)
    t0 = 1_700_000_000.0
    s.samples = [(t0 - 0.5, 1200.0, 2070.0, 0), (t0 + 0.002, 2070.0, 2070.0, 0),
                 (t0 + 0.004, 2040.0, 2070.0, 0x4), (t0 + 0.006, 2070.0, 2070.0, 0),
                 (t0 + 1.0, 900.0, 2070.0, 0x40)]
    c = s.summary(t0, t0 + 0.008)
    assert c["samples"] == 3 and c["sm_mhz"] == 2070 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"] and c["source"] == "nvml"
    c2 = s.summary(t0 + 0.9, t0 + 1.1)
    assert c2["reasons"] == ["hw_thermal_slowdown"]

"""Host logic of bench.py that needs no GPU: the clock samples behind the timing rules.

A run is rejected when its timed region saw hw_slowdown, hw_thermal_slowdown or
sw_thermal_slowdown, or SM clocks stuck below the maximum; the bench reports each
region's median SM clock, maximum clock, median power and the reasons seen in it.
These tests feed the parser an nvidia-smi CSV written here and bin it by time.
"""
import datetime

import bench


def _line(t, sm, power="950.00", reasons=("Not Active",) * 4):
    stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return ", ".join([stamp, "0", str(sm), "2032", power, "0x0000000000000004", *reasons]) + "\n"


def _sampler(tmp_path, lines):
    path = tmp_path / "clocks.csv"
    path.write_text("".join(lines))
    c = bench.ClockSampler(0)
    c.proc = object()  # as if nvidia-smi had run
    c.samples = bench.ClockSampler.parse(str(path))
    return c


def test_region_bins_samples_by_time(tmp_path):
    t0 = 1_700_000_000.0
    cap = ("Not Active", "Not Active", "Not Active", "Active")
    lines = [_line(t0 + 0.025 * i, 1900) for i in range(4)]                        # warm-up, idle clock
    lines += [_line(t0 + 0.1 + 0.025 * i, 1500 + i, reasons=cap) for i in range(5)]  # timed region
    lines += [_line(t0 + 0.3, 1700, power="[N/A]")]
    lines += ["garbage line\n", "2024/01/01, 0, x, y, z, 0, a, b, c, d\n"]           # skipped
    c = _sampler(tmp_path, lines)
    assert len(c.samples) == 10
    r = c.region(t0 + 0.09, t0 + 0.21)
    assert r["samples"] == 5 and r["sm_mhz"] == 1502 and r["sm_max_mhz"] == 2032.0
    assert r["reasons"] == ["sw_power_cap"] and r["power_w"] == 950.0
    w = c.region(t0 - 1, t0 + 0.08)
    assert w["sm_mhz"] == 1900 and w["reasons"] == []
    n = c.region(t0 + 0.29, t0 + 0.31)  # power not available: median of none
    assert n["sm_mhz"] == 1700 and n["power_w"] is None


def test_rejecting_reasons_are_reported(tmp_path):
    t0 = 1_700_000_100.0
    lines = [_line(t0, 1400, reasons=("Active", "Not Active", "Not Active", "Not Active")),
             _line(t0 + 0.025, 1400, reasons=("Not Active", "Active", "Not Active", "Active"))]
    r = _sampler(tmp_path, lines).region(t0 - 0.01, t0 + 0.05)
    assert r["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap"]


def test_unsampled_region():
    c = bench.ClockSampler(0)
    r = c.region(0.0, 1.0)
    assert r["sm_mhz"] is None and r["reasons"] == ["unsampled"]

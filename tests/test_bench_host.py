"""Host logic of the benchmark that needs no GPU: the clock record kept beside every
number (samples of nvidia-smi inside the timed region only, median SM clock, the throttle
reasons that were active)."""
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _stamp(t):
    return time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(t)) + ".%03d" % int(round((t % 1) * 1000) % 1000)


def _line(t, mhz, reasons=()):
    flags = ["Active" if n in reasons else "Not Active" for n in bench.REASON_NAMES]
    return ", ".join([_stamp(t), "0", str(mhz), "2070", "900.00", "0x0"] + flags)


def test_clock_samples_inside_the_timed_region_only():
    t = 1_800_000_000.25
    lines = [_line(t - 2.0, 300, ("hw_slowdown",)),  # before the region: idle clock, a slowdown
             _line(t + 0.1, 2070), _line(t + 0.2, 2060, ("sw_power_cap",)), _line(t + 0.3, 2070),
             _line(t + 3.0, 1200, ("sw_thermal_slowdown",)),  # after it
             "garbage, line", ""]
    got = bench.parse_clock_samples(lines, t, t + 1.0)
    assert got == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    every = bench.parse_clock_samples(lines)
    assert every["samples"] == 5 and every["reasons"] == ["hw_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    assert bench.parse_clock_samples(lines, t + 5, t + 6)["samples"] == 0

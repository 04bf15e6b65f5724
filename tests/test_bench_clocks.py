"""bench.py's clock record: only nvidia-smi samples taken inside the timed region count (CPU, fake lines)."""
import time

import bench


def _line(t, sm, reasons=("Not Active",) * 4):
    stamp = time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(int(t))) + f".{int(round((t % 1) * 1000)):03d}"
    return ", ".join([stamp, "0", str(sm), "2070", "900.5", "0x0000000000000000", *reasons])


def test_only_samples_inside_the_timed_region_count():
    t0 = 1_800_000_000.0
    lines = [_line(t0 - 0.30, 1000), _line(t0 - 0.10, 1005)]                      # idle, before
    lines += [_line(t0 + 0.02 * i, 2070 - i) for i in range(1, 6)]                 # inside
    lines += [_line(t0 + 0.50, 900, ("Not Active", "Active", "Not Active", "Not Active"))]   # after
    r = bench.summarize_clock_lines(lines, t0, t0 + 0.11, 20)
    assert r["samples"] == 5
    assert r["sm_mhz"] == 2067.0
    assert r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == []
    assert r["window"] == "timed region"


def test_throttle_reasons_inside_the_region_are_reported():
    t0 = 1_800_000_000.0
    lines = [_line(t0 + 0.01, 1800, ("Not Active", "Not Active", "Not Active", "Active")),
             _line(t0 + 0.03, 1700, ("Active", "Not Active", "Not Active", "Not Active"))]
    r = bench.summarize_clock_lines(lines, t0, t0 + 0.05, 20)
    assert r["samples"] == 2 and r["sm_mhz"] == 1750.0
    assert r["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_malformed_lines_are_skipped_and_no_timestamps_fall_back_to_all():
    lines = ["garbage", "1, 2, 3", "not-a-time, 0, 1900, 2070, 1.0, 0x0, Not Active, Not Active, Not Active, "
             "Not Active"]
    r = bench.summarize_clock_lines(lines, 0.0, 1.0, 20)
    assert r["samples"] == 1 and r["sm_mhz"] == 1900.0
    assert r["window"] == "whole run (no timestamps)"

"""The benchmark's clock record on CPU: nvidia-smi lines (ClockSampler.FIELDS)
are reduced to the median SM clock, the largest max clock and the throttle
reasons of the samples taken inside the timed region only."""
import datetime

import bench


def _line(t, sm, mx=2070, reasons=("Not Active",) * 4):
    ts = t.strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return ", ".join([ts, "0", str(sm), str(mx), "900.00", "0x0000000000000000", *reasons])


def test_only_samples_inside_the_region_count():
    t0 = datetime.datetime(2026, 1, 1, 12, 0, 0)
    lines = [_line(t0 - datetime.timedelta(milliseconds=200), 345),          # idle, before
             _line(t0 + datetime.timedelta(milliseconds=100), 2070),
             _line(t0 + datetime.timedelta(milliseconds=300), 2055,
                   reasons=("Not Active", "Not Active", "Not Active", "Active")),
             _line(t0 + datetime.timedelta(milliseconds=500), 2070),
             _line(t0 + datetime.timedelta(milliseconds=900), 300)]            # idle, after
    r = bench.parse_clock_lines(lines, t0, t0 + datetime.timedelta(milliseconds=600))
    assert r == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    # a region shorter than the sampling interval keeps every sample
    r = bench.parse_clock_lines(lines, t0 + datetime.timedelta(milliseconds=101),
                                t0 + datetime.timedelta(milliseconds=102))
    assert r["samples"] == 5
    assert bench.parse_clock_lines(["garbage", ""]) is None


def test_fields_match_the_parser():
    # timestamp first, then index, clocks.sm, clocks.max.sm, power, active, four reasons
    assert bench.ClockSampler.FIELDS.split(",")[0] == "timestamp"
    assert len(bench.ClockSampler.FIELDS.split(",")) == 10

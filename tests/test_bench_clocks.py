"""The benchmark's clock record on CPU: nvidia-smi samples summarised into the median SM clock
under load and the throttle reasons seen (a run with a hardware or thermal slowdown is
rejected, so the parse must not miss one)."""

import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402

NA, ACT = "Not Active", "Active"


def _line(sm, mx, hw=NA, hwt=NA, swt=NA, cap=NA, util=100):
    return f"{sm}, {mx}, {hw}, {hwt}, {swt}, {cap}, {util}"


def test_median_under_load_and_no_reasons():
    out = "\n".join([_line(600, 2070, util=0), _line(2070, 2070), _line(2040, 2070), _line(2070, 2070),
                     _line(1980, 2070)])
    d = bench.ClockSampler.summarize(out)
    assert d["sm_mhz"] == 2070.0 and d["sm_max_mhz"] == 2070.0 and d["reasons"] == []
    assert d["samples"] == 5 and d["samples_under_load"] == 4


def test_reasons_seen_under_load_are_reported():
    out = "\n".join([_line(1800, 2070, cap=ACT), _line(1700, 2070, hwt=ACT), _line(2070, 2070),
                     _line(500, 2070, hw=ACT, util=0)])
    d = bench.ClockSampler.summarize(out)
    assert d["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]  # the idle sample's is not under load
    assert d["sm_mhz"] == 1800.0


def test_idle_only_and_garbage_lines():
    d = bench.ClockSampler.summarize("garbage\n" + _line(1200, 2070, util=0) + "\n[N/A], 2070, x, x, x, x, 0\n")
    assert d["sm_mhz"] == 1200.0 and d["samples_under_load"] == 0
    assert bench.ClockSampler.summarize("")["reasons"] == ["no samples"]

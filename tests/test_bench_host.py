"""Host-side logic of bench.py (no GPU): the clock record and the workload
overrides."""

import datetime
import importlib.util
import os
import sys

import pytest

from workloads import configs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_host", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


class _FakeSmi:
    """Stands in for the nvidia-smi process: canned samples."""

    def __init__(self, lines):
        self.lines = lines

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return "".join(self.lines), ""


def _line(t, sm, reason_cap="Not Active", thermal="Not Active"):
    return "%s, %d, 2070, 0x0, Not Active, Not Active, %s, %s\n" % (t, sm, thermal, reason_cap)


def test_clock_samples_kept_inside_the_window():
    b = _bench()
    c = b.Clocks(0)
    c.first = _line("2026/12/02 11:13:05.100", 1500)                 # start-up, before the window
    c.proc = _FakeSmi([_line("2026/12/02 11:13:05.300", 2070),
                       _line("2026/12/02 11:13:05.500", 2050, reason_cap="Active"),
                       _line("2026/12/02 11:13:06.900", 1200, thermal="Active")])   # after it
    c.mark(datetime.datetime(2026, 12, 2, 11, 13, 5, 200000), datetime.datetime(2026, 12, 2, 11, 13, 5, 600000))
    r = c.stop()
    assert r == {"sm_mhz": 2060.0, "sm_max_mhz": 2070.0, "samples": 2, "reasons": ["sw_power_cap"]}


def test_clock_window_shorter_than_the_period():
    # no sample inside: the two around the window stand for it
    b = _bench()
    c = b.Clocks(0)
    c.first = _line("2026/12/02 11:13:05.100", 2000)
    c.proc = _FakeSmi([_line("2026/12/02 11:13:05.300", 2070), _line("2026/12/02 11:13:05.500", 1000)])
    c.mark(datetime.datetime(2026, 12, 2, 11, 13, 5, 150000), datetime.datetime(2026, 12, 2, 11, 13, 5, 170000))
    r = c.stop()
    assert r["samples"] == 2 and r["sm_mhz"] == 2035.0


def test_clock_unreadable_stamps_are_kept():
    b = _bench()
    c = b.Clocks(0)
    c.proc = _FakeSmi(["n/a, 2070, 2070, 0x0, Not Active, Not Active, Not Active, Not Active\n"])
    c.mark(datetime.datetime(2026, 12, 2), datetime.datetime(2026, 12, 2))
    assert c.stop()["samples"] == 1


def test_workload_overrides():
    b = _bench()
    saved = sys.argv
    try:
        sys.argv = ["bench.py", "--ubatch", "128"]
        cfg = b.apply_overrides(configs.config(2), b.parse())
        assert cfg["params"]["n_ubatch"] == 128 and cfg["name"].endswith("-ub128")
        assert "-ub512" not in cfg["name"]
        sys.argv = ["bench.py", "--config", "3", "--streams", "8", "--kv-per-stream", "4096"]
        cfg = b.apply_overrides(configs.config(3), b.parse())
        assert (cfg["params"]["n_stream"], cfg["params"]["n_ctx"]) == (8, 32768)
        sys.argv = ["bench.py"]
        cfg = b.apply_overrides(configs.config(2), b.parse())
        assert cfg == configs.config(2)
    finally:
        sys.argv = saved


@pytest.mark.parametrize("cid", [2, 3, 4, 5])
def test_counted_work_is_positive(cid):
    # the bookkeeping behind the roofline: tokens per step for every workload
    b = _bench()
    assert b.measured_tokens(configs.config(cid)) > 0

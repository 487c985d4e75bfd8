"""Host logic of the benchmark that needs no GPU: the clock record (samples
kept to the timed region, throttle reasons), the early-exit byte accounting,
and the default step counts of the two arms."""
import datetime
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _line(ts, sm, mx=2070, reasons=("Not Active",) * 4):
    return ", ".join([ts.strftime("%Y/%m/%d %H:%M:%S.%f")[:-3], "0", str(sm), str(mx), "900.0",
                      "0x0", *reasons])


def test_clock_record_keeps_the_timed_region():
    c = bench.Clocks(0)
    t0 = datetime.datetime(2026, 1, 2, 3, 4, 5, 0)
    c.t0, c.t1 = t0 + datetime.timedelta(milliseconds=100), t0 + datetime.timedelta(milliseconds=200)
    c.lines = [_line(t0, 1000),                                            # before: idle
               _line(t0 + datetime.timedelta(milliseconds=120), 2070),
               _line(t0 + datetime.timedelta(milliseconds=140), 2055),
               _line(t0 + datetime.timedelta(milliseconds=160), 2070,
                     reasons=("Not Active", "Not Active", "Not Active", "Active")),
               _line(t0 + datetime.timedelta(milliseconds=300), 800,
                     reasons=("Active", "Not Active", "Not Active", "Not Active"))]  # after
    s = c.summary()
    assert s["samples_in_timed_region"] == 3 and s["samples"] == 3
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]      # the hw_slowdown sample lies outside


def test_clock_record_falls_back_to_all_samples():
    c = bench.Clocks(0)
    t0 = datetime.datetime(2026, 1, 2, 3, 4, 5, 0)
    c.t0 = c.t1 = t0 + datetime.timedelta(seconds=5)   # no sample inside
    c.lines = [_line(t0, 1500), _line(t0 + datetime.timedelta(milliseconds=20), 1700),
               "garbage line"]
    s = c.summary()
    assert s["samples_in_timed_region"] == 0 and s["samples"] == 2 and s["sm_mhz"] == 1600.0
    c.lines = []
    assert c.summary()["reasons"] == ["unsampled"]


class _Wl:
    """The parts of a workload that the byte accounting reads."""
    def __init__(self, early, greedy=False):
        self.early, self.greedy, self.V, self.esize = early, greedy, 1000, 2
        self.rounds = [dict(depth=np.full(4, 7, np.int64))]


def test_early_exit_bytes_follow_the_walk():
    acc = np.array([0, 3, 7, 6])          # a < 7: 2(a + 1) rows; a = 7: 15 rows
    rows = 2 * 1 + 2 * 4 + 15 + 2 * 7
    assert bench.Workload.stats_bytes(_Wl(True), 0, acc) == rows * 1000 * 2
    assert bench.Workload.stats_bytes(_Wl(False), 0, acc) == 4 * 15 * 1000 * 2
    assert bench.Workload.stats_bytes(_Wl(False, greedy=True), 0) == 4 * 8 * 1000 * 2


def test_default_steps_per_arm(monkeypatch):
    seen = {}
    monkeypatch.setattr(bench, "run_reference", lambda a: seen.setdefault("ref", a.steps))
    monkeypatch.setattr(bench, "run_ours", lambda a: seen.setdefault("ours", a.steps))
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference"])
    bench.main()
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    bench.main()
    assert seen == {"ref": 20, "ours": 1000}
    monkeypatch.setattr(sys, "argv", ["bench.py", "--steps", "7"])
    seen.pop("ours")
    bench.main()
    assert seen == {"ref": 20, "ours": 7}

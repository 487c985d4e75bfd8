"""Host logic of the benchmark that needs no GPU: the clock record (samples
kept to the timed region, throttle reasons), the early-exit byte accounting,
the default step counts of the two arms, and the reference arm's line."""
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


def test_reference_arm_prints_the_contract_line(monkeypatch, capsys):
    """The reference arm (the CPU oracle) on the small chain: one JSON line
    with the keys of the benchmark contract, its own cpu_baseline and an e2e
    with no host-device traffic."""
    import json
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--config", "1",
                                      "--steps", "2", "--warmup", "1", "--cpu-sample", "2"])
    bench.main()
    out = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(out) == 1
    line = json.loads(out[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 1
    assert line["value"] > 0 and line["unit"] == "rows/s" and line["higher_is_better"] is True
    assert line["config"]["workload"].startswith("config 1")
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "rows/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


_SECONDARY_KEYS = ("value", "unit", "steps", "ms_per_step", "accepted_tokens_per_s",
                   "mean_accept_len", "rows_read_per_s", "hbm_gbs", "hbm_frac_measured",
                   "roofline", "kernels", "repeats", "clocks", "alg_bytes_per_step", "config")


def test_secondary_lines_only_on_the_default_run(monkeypatch, capsys):
    """The default run (config 5) adds the large-vocabulary chain's full and
    early-exit lines, each over at least SECONDARY_STEPS device-resident
    steps; a flag that changes the workload, or --no-secondary, leaves them
    out."""
    import json
    import torch
    calls = []

    def fake_measure(a, rank, world, local):
        calls.append((a.config, a.early_exit, a.steps, a.no_e2e, a.no_cpu_baseline))
        return {k: a.config for k in _SECONDARY_KEYS}

    monkeypatch.setattr(bench, "measure", fake_measure)
    monkeypatch.setattr(torch.cuda, "set_device", lambda *a, **k: None)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--steps", "7"])
    bench.main()
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert calls == [(5, False, 7, False, False),
                     (3, False, bench.SECONDARY_STEPS, True, True),
                     (3, True, bench.SECONDARY_STEPS, True, True)]
    assert sorted(line["secondary"]) == ["config 3: large_vocab_chain",
                                         "config 3: large_vocab_chain (early exit)"]
    assert all(set(v) == set(_SECONDARY_KEYS) for v in line["secondary"].values())
    for extra in (["--no-secondary"], ["--greedy"], ["--config", "3"]):
        calls.clear()
        monkeypatch.setattr(sys, "argv", ["bench.py", "--steps", "7", *extra])
        bench.main()
        line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
        assert len(calls) == 1 and "secondary" not in line, extra

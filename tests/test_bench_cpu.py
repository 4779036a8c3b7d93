"""bench.py helpers that need no GPU: default arguments within the timing rules, the config
line, and the single-thread oracle timing of the tiny configuration reported beside the CPU
baseline."""
import sys

import bench
import synth


def test_defaults_follow_the_timing_rules(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse()
    assert a.gpus == 1 and a.warmup >= 3 and a.steps >= 50 and a.e2e_steps >= 50
    assert a.impl == "mageflow" and a.workload == "native16k"


def test_config_line_names_the_workload():
    c = bench.config_dict(synth.FULL)
    assert "workload" in c and c["budget"] == 16384 and c["hidden"] == 3072 and "l2" in c


def test_tiny_single_thread_timing():
    tps, n = bench.tiny_single_thread(0.05)
    assert tps > 0 and n >= 1

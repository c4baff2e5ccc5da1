"""The bench's reference arm (the oracle on bounded row samples) on a small stand-in
configuration: one JSON line with the contract's keys, rank 0 only (CPU)."""
import argparse
import dataclasses
import json

import pytest

import bench
import dsa_workloads as W


@pytest.fixture
def small_prefill(monkeypatch):
    # the prefill_4k name, with the tiny configuration's sizes, so the oracle finishes fast
    cfg = dataclasses.replace(W.CONFIGS["tiny"], name="prefill_4k")
    monkeypatch.setitem(W.CONFIGS, "prefill_4k", cfg)
    return cfg


def test_reference_arm_prints_one_line(small_prefill, capsys):
    args = argparse.Namespace(workload="prefill_4k", steps=2, warmup=1)
    bench.run_reference(args, rank=0, world=1)
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_do_nothing(small_prefill, capsys):
    args = argparse.Namespace(workload="prefill_4k", steps=2, warmup=1)
    bench.run_reference(args, rank=1, world=2)
    assert capsys.readouterr().out == ""

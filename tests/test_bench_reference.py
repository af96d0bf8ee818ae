"""bench.py's reference arm (the oracle on the host cores) on the CPU: one JSON
line carrying the keys the benchmark contract asks for, with values that agree
with each other.  No GPU."""
import argparse

import pytest

import bench

CONTRACT_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                 "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"}


def _args(**kw):
    a = dict(gpus=1, steps=2, warmup=1, impl="reference", workload="tiny_fp32", tokens=16, replicas=0,
             no_cpu_baseline=False, sweep=False, eager=False)
    a.update(kw)
    return argparse.Namespace(**a)


def test_reference_line_has_the_contract_keys():
    line = bench.run_reference(_args(), 0, 1)
    assert CONTRACT_KEYS <= set(line)
    assert line["impl"] == "reference"
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["unit"] == "tokens/s" and line["e2e"]["unit"] == "tokens/s"
    # one token per step: tokens/s and ms per step describe the same timing
    assert line["value"] == pytest.approx(1e3 / line["ms_per_step"], rel=1e-2)
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"].startswith("tiny_fp32")


def test_reference_arm_runs_on_rank_zero_only():
    assert bench.run_reference(_args(), 1, 2) is None

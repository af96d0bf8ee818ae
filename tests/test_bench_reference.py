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


def test_routing_stats_of_uniform_and_zipf_loads():
    import json

    import numpy as np
    E = 128
    flat = bench.routing_stats(np.repeat(np.arange(E), 6).reshape(-1, 6), E)
    assert flat["experts_with_routes"] == E and flat["max_over_mean"] == 1.0
    assert flat["cv2"] == 0.0 and flat["norm_entropy"] == 1.0 and flat["loglog_slope"] is None
    # 6 rows per expert in 128-row tiles: 122 of every 128 rows are padding
    assert flat["tail_waste_128_row_tiles"] == round(1 - 6 / 128, 3)
    rng = np.random.default_rng(0)
    w = 1.0 / np.arange(1, E + 1) ** 1.1
    ids = rng.choice(E, size=(20000, 1), p=w / w.sum())
    z = bench.routing_stats(ids, E)
    assert -1.3 < z["loglog_slope"] < -0.9          # about -s for Zipf(s = 1.1)
    assert z["max_over_mean"] > 10 and 0.5 < z["norm_entropy"] < 0.9
    json.dumps(z)                                    # plain JSON types


def test_roofline_numerators_match_the_worked_ledgers():
    """The bench's algorithmic bytes and FLOPs per step against the per-unit
    figures worked out by hand for the five workloads: one Nano expert is
    2 x 1856 x 2688 x 2 B, one Super NVFP4 expert block 3,096,576 B (page
    "Nemotron-3.5-Super 120B on an 8 GB GPU") plus its two FP32 tensor scales."""
    from synth import NANO_DECODE, SUPER_LATENT, SUPER_NVFP4, TINY_FP32
    nano = bench.layer_bytes(NANO_DECODE, 6, 1)
    assert nano["experts"] == 6 * 19_955_712
    assert nano["shared"] == 39_911_424 and nano["router"] == 1_376_768
    assert nano["total"] == 161_033_216
    sup = bench.layer_bytes(SUPER_LATENT, 22, 1)
    assert sup["experts"] == 22 * 11_010_048 and sup["shared"] == 88_080_384
    assert sup["latent"] == 16_777_216 and sup["router"] == 8_390_656
    assert sup["total"] == 355_485_696
    fp4 = bench.layer_bytes(SUPER_NVFP4, 22, 1)
    assert fp4["experts"] == 22 * (3_096_576 + 8)
    assert fp4["total"] == 181_389_488
    assert bench.layer_flops(SUPER_LATENT, 1) == 351_272_960
    assert bench.layer_flops(TINY_FP32, 16) == 16 * 528_384


def test_recorded_traffic_is_reported_only_for_unchanged_sources(tmp_path, monkeypatch):
    """The roofline `traffic` comes from the committed ncu table only while the
    kernel family's sources hash to the value recorded beside it."""
    want = bench.sources_sha16("gemv")
    assert len(want) == 16 and int(want, 16) >= 0
    table = tmp_path / "traffic.md"
    table.write_text("| kernel | workload | dram bytes per launch | sources sha16 |\n|---|---|---|---|\n"
                     f"| `k<0>` | w T=1 | 1,234,000 | {want} |\n"
                     "| `k<1>` | w T=1 | 5,678,000 | 0000000000000000 |\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(table))
    assert bench.recorded_traffic("k<0>", "w T=1", "gemv") == (1234000, want)
    assert bench.recorded_traffic("k<1>", "w T=1", "gemv") == (None, "0000000000000000")
    assert bench.recorded_traffic("k<2>", "w T=1", "gemv") == (None, None)


def test_committed_traffic_rows_parse():
    """Every row of the committed table names a kernel, a workload, a byte
    count and a 16-digit source hash (whether or not it is current)."""
    rows = 0
    for line in open(bench.TRAFFIC_FILE):
        cells = [c.strip().strip("`") for c in line.strip().strip("|").split("|")]
        if len(cells) == 4 and cells[3] and all(ch in "0123456789abcdef" for ch in cells[3]) and len(cells[3]) == 16:
            assert int(cells[2].replace(",", "")) > 0
            rows += 1
    assert rows >= 1

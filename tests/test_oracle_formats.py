"""Pins for the oracle's number formats (BF16 rounding, E2M1, E4M3, NVFP4 layout)
and for the workload shapes through the byte counts the pages print."""
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from synth import NANO_DECODE, SUPER_LATENT, quantize_nvfp4

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _golden_kv(name):
    out = {}
    for line in open(os.path.join(GOLD, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, v = line.split()
        out[k] = float(v)
    return out


# ---------------------------------------------------------------- BF16 ------
def test_bf16_round_matches_torch_cast_of_fp32_values():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.0e38, -2.5e-39, 1e-45])])
    v32 = v.astype(np.float32)
    ref = torch.from_numpy(v32).to(torch.bfloat16).float().numpy().astype(np.float64)
    got = O.bf16_round(v32.astype(np.float64))
    assert np.array_equal(np.nan_to_num(ref, posinf=9e99, neginf=-9e99),
                          np.nan_to_num(got, posinf=9e99, neginf=-9e99))


def test_bf16_round_ties_to_even_and_keeps_eight_bits():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: the even neighbour is 1
    assert O.bf16_round(1.0 + 2.0 ** -8) == 1.0
    # 1 + 3*2^-8 is halfway between 1+2^-7 and 1+2^-6: the even neighbour is 1+2^-6
    assert O.bf16_round(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    # 255 and 257: 8 significant bits hold 255 exactly, 257 rounds to 256
    assert O.bf16_round(255.0) == 255.0 and O.bf16_round(257.0) == 256.0
    # rounding straight from float64 (one rounding) differs from going through FP32
    x = 1.0 + 2.0 ** -8 + 2.0 ** -40       # just above the midpoint
    assert O.bf16_round(x) == 1.0 + 2.0 ** -7


# ---------------------------------------------------------------- E2M1 ------
def test_e2m1_table_is_the_nvfp4_value_set():
    mags = [O.e2m1_value(c) for c in range(8)]
    assert mags == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert [O.e2m1_value(c | 8) for c in range(1, 8)] == [-m for m in mags[1:]]


def test_e4m3_decode_matches_torch_float8_for_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = np.array([O.e4m3_value(b) for b in range(256)])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    assert np.nanmax(got) == 448.0 and O.e4m3_value(1) == 2.0 ** -9


def test_nvfp4_round_trip_of_representable_values_is_exact():
    # values E2M1 * 448 * 2^-9: every block holds a 6 (block scale 448, the
    # largest E4M3 value) and the tensor amax 5.25 gives the exact per-tensor
    # scale 2^-9, so quantising and dequantising must return them unchanged
    rng = np.random.default_rng(1)
    N, K = 8, 64
    codes = rng.integers(0, 16, size=(N, K))
    codes[:, ::16] = 7                      # each block holds a +6 (its amax)
    vals = np.array([[O.e2m1_value(int(c)) for c in row] for row in codes]) * 448.0 * 2.0 ** -9
    w = torch.from_numpy(vals.astype(np.float32)).to(torch.bfloat16)
    q, sf, gs = quantize_nvfp4(w)
    back = O.dequant_nvfp4(q.numpy(), sf.numpy(), gs.numpy())
    np.testing.assert_array_equal(back, vals)


def test_nvfp4_nibble_order_matters():
    # the even element sits in the low nibble; swapping the halves must be caught
    rng = np.random.default_rng(2)
    w = torch.from_numpy(rng.standard_normal((4, 64)).astype(np.float32)).to(torch.bfloat16)
    q, sf, gs = quantize_nvfp4(w)
    good = O.dequant_nvfp4(q.numpy(), sf.numpy(), gs.numpy())
    swapped = ((q >> 4) | (q << 4)).numpy().astype(np.uint8)
    bad = O.dequant_nvfp4(swapped, sf.numpy(), gs.numpy())
    err_good = np.abs(good - w.float().numpy()).max()
    err_bad = np.abs(bad - w.float().numpy()).max()
    assert err_good < 0.2 * np.abs(w.float().numpy()).max()
    assert err_bad > 3 * err_good


def test_nvfp4_quantisation_error_is_within_half_a_step():
    rng = np.random.default_rng(3)
    w32 = rng.standard_normal((16, 128)).astype(np.float32)
    w = torch.from_numpy(w32).to(torch.bfloat16)
    q, sf, gs = quantize_nvfp4(w)
    back = O.dequant_nvfp4(q.numpy(), sf.numpy(), gs.numpy())
    wf = w.float().numpy()
    scale = np.repeat(np.array([[O.e4m3_value(int(b)) for b in row] for row in sf.numpy()]), 16, axis=-1) * float(gs)
    # largest E2M1 gap is 2 (between 4 and 6); rounding error <= gap/2 * scale,
    # plus saturation when the E4M3 block scale rounded down (<= 1/16 of amax)
    assert np.all(np.abs(back - wf) <= 1.0 * scale + np.abs(wf) / 16 + 1e-12)


# ----------------------------------------------------- byte-count pins ------
def test_super_nvfp4_expert_block_is_3096576_bytes():
    g = _golden_kv("byte_ledgers.txt")
    s = SUPER_LATENT
    one_up = torch.zeros((s.d_expert, s.d_e), dtype=torch.bfloat16)
    one_down = torch.zeros((s.d_e, s.d_expert), dtype=torch.bfloat16)
    qu, su, _ = quantize_nvfp4(one_up)
    qd, sd, _ = quantize_nvfp4(one_down)
    up_bytes = qu.numel() + su.numel()
    total = up_bytes + qd.numel() + sd.numel()
    assert total == g["nvfp4_expert_block_bytes"]
    assert round(up_bytes / 1e6, 2) == g["nvfp4_expert_up_mb"]
    per_token = s.top_k * g["super_moe_layers"] * total / 1e9
    assert abs(per_token - g["super_routed_per_token_gb_approx"]) < 0.05
    assert abs(per_token - g["super_routed_gb"]) < 0.006


def test_nano_bf16_expert_and_shared_bytes_match_the_lightning_ledger():
    g = _golden_kv("byte_ledgers.txt")
    s = NANO_DECODE
    expert = 2 * s.d_model * s.d_expert * 2          # up + down, BF16
    shared = 2 * s.d_model * s.d_shared * 2
    # the page's two figures share the layer count: their ratio fixes K*expert/shared
    # (both are printed to 0.01 GB, so the ratio is known to an interval)
    ex, sh = g["lightning_experts_gb"], g["lightning_shared_gb"]
    assert (ex - 0.005) / (sh + 0.005) <= s.top_k * expert / shared <= (ex + 0.005) / (sh - 0.005)
    # with 23 MoE layers (the Lightning layer count) both round to the printed values
    assert round(23 * s.top_k * expert / 1e9, 2) == g["lightning_experts_gb"]
    assert round(23 * shared / 1e9, 2) == g["lightning_shared_gb"]


def test_super_latent_pair_and_shared_bytes_match_the_super_ledger():
    g = _golden_kv("byte_ledgers.txt")
    s = SUPER_LATENT
    layers = g["super_moe_layers"]
    latent_pair = 2 * s.d_model * s.d_latent * 2
    assert round(layers * latent_pair / 1e9, 2) == g["super_latent_pair_gb"]
    shared_nvfp4 = 2 * s.d_model * s.d_shared * (0.5 + 1 / 16)
    assert round(layers * shared_nvfp4 / 1e9, 2) == g["super_shared_nvfp4_gb"]

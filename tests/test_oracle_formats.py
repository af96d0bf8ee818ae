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


# ------------------------------------------------ NVFP4 activation terms ----
def test_e4m3_rn_code_matches_torch_cast():
    """Round-to-nearest-even onto E4M3 (saturating at 448) equals torch's
    float8_e4m3fn cast on random values, subnormals and exact midpoints."""
    rng = np.random.default_rng(3)
    grid = np.array([O.e4m3_value(b) for b in range(127)])
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
    v = np.concatenate([rng.uniform(0, 448, 5000), 2.0 ** rng.uniform(-12, 8.8, 5000), mids, grid,
                        [0.0, 448.0, 2.0 ** -10, 3 * 2.0 ** -11]]).astype(np.float32)
    v = v[v <= 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_rn_code(v), ref)
    assert O.e4m3_rn_code(np.float32(1e6)) == 126            # saturates to 448


def test_e2m1_rn_code_matches_the_weight_quantiser():
    """Signed E2M1 rounding equals the synthetic weights' encoder (ties to the
    even code, saturating at 6) on random values and every midpoint."""
    from synth.generate import _e2m1_codes
    rng = np.random.default_rng(4)
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    v = np.concatenate([rng.uniform(-8, 8, 20000), mids, [-m for m in mids], [0, 6, -6, 7.5, -100]]).astype(np.float32)
    ref = _e2m1_codes(torch.from_numpy(v)).numpy()
    assert np.array_equal(O.e2m1_rn_code(v), ref)


def test_first_activation_term_is_the_weight_quantiser():
    """One term of a row is the NVFP4 encoding the synthetic weights use
    (per-row scale amax/(6*448), E4M3 block scales, E2M1 codes): scales
    exactly; values exactly except where the weight encoder's r / s and the
    activation quantiser's r * (1/s) fall on the two sides of an E2M1
    rounding boundary (the two FP32 ratios differ by at most 2 ulp)."""
    rng = np.random.default_rng(5)
    x = torch.from_numpy(rng.standard_normal((6, 256)).astype(np.float32) * 3).to(torch.bfloat16).float()
    codes, sf, g = O.nvfp4_terms(x.numpy(), 1)
    grid = np.array([O.e2m1_value(i) for i in range(8)])
    mids = (grid[1:] + grid[:-1]) / 2
    val = lambda c: np.where(c & 8, -1.0, 1.0) * grid[c & 7]
    n_diff = 0
    for t in range(6):
        q, s, gs = quantize_nvfp4(x[t:t + 1])
        ref_codes = np.empty(256, dtype=np.uint8)
        ref_codes[0::2] = q.numpy()[0] & 0xF
        ref_codes[1::2] = q.numpy()[0] >> 4
        assert np.array_equal(sf[0, t], s.numpy()[0])
        assert g[t] == np.float32(gs.item())
        diff = np.where(val(codes[0, t]) != val(ref_codes))[0]
        n_diff += diff.size
        for k in diff:                      # only at a rounding boundary
            scale = np.float32(O.e4m3_value(int(sf[0, t, k // 16])) * np.float32(g[t]))
            ratio = abs(float(x[t, k]) / float(scale))
            assert np.min(np.abs(mids - ratio)) <= 4 * np.finfo(np.float32).eps * ratio
    assert n_diff <= 3


def test_activation_terms_of_representable_values():
    """Blocks that are powers of two times E2M1 values come back from the
    first term exactly (codes) and the remaining residual is FP32 noise."""
    rng = np.random.default_rng(6)
    vals = np.array([O.e2m1_value(c) for c in range(16)])
    x = np.empty((2, 128), dtype=np.float32)
    for t in range(2):
        for b in range(8):
            blk = rng.choice(vals, 16)
            blk[0] = 6.0                                   # every block reaches the top code
            x[t, 16 * b:16 * b + 16] = blk * 2.0 ** (b - 4)
    codes, sf, g = O.nvfp4_terms(x, 3)
    c0 = np.where(codes[0] & 8, -1.0, 1.0) * np.abs(vals[codes[0] & 7])
    expect = x.reshape(2, 8, 16) / (2.0 ** (np.arange(8) - 4))[None, :, None]
    assert np.array_equal(c0.reshape(2, 8, 16), expect)
    rec = O.dequant_terms(codes, sf, g)
    assert np.max(np.abs(rec - x)) <= 1e-6 * np.max(np.abs(x))


def test_activation_terms_shrink_the_error_per_term():
    """Each term leaves at most ~0.18 of the previous residual of a block (the
    E2M1 grid's widest half-gap relative to its top value, plus the E4M3 scale
    rounding), so n terms reach 0.18^n of the block's largest magnitude."""
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((8, 1024)) * np.exp(rng.standard_normal((8, 1)))).astype(np.float32)
    bmax = np.abs(x.reshape(8, 64, 16)).max(-1)
    prev = None
    for n in (1, 2, 3, 4):
        err = np.abs(O.nvfp4_activations(x, n) - x).reshape(8, 64, 16).max(-1)
        assert np.all(err <= 0.18 ** n * bmax + 1e-30)
        if prev is not None:
            assert err.max() < prev
        prev = err.max()


def test_many_activation_terms_converge_to_the_exact_mlp():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((5, 256))
    up = rng.standard_normal((128, 256)) / 16
    down = rng.standard_normal((256, 128)) / 11
    exact = O.relu2_mlp(x, up, down, bf16_points=False)
    approx = O.relu2_mlp(x, up, down, bf16_points=False, act_terms=6)
    assert np.max(np.abs(approx - exact)) <= 1e-4 * np.sqrt(np.mean(exact ** 2))
    # one term (plain W4A4) quantises both product inputs: x and h
    xq = O.nvfp4_activations(x, 1)
    h = O.nvfp4_activations(np.maximum(xq @ up.T, 0) ** 2, 1)
    assert np.allclose(O.relu2_mlp(x, up, down, bf16_points=False, act_terms=1), h @ down.T, rtol=0, atol=1e-12)

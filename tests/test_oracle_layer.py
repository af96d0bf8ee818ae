"""Pins for the oracle's expert MLP and the whole layer.

No page prints a worked layer output for NemotronH shapes, so the layer is
pinned by hand-computed MLP values, by the identity that a one-expert top-1
layer is a scaled dense ReLU^2 MLP, by a token-major schedule (page "Nemotron
Is Not One Circuit", section "Routing Is Cheap; Expert Memory Is The Hard
Part": the token-major reference) checked against the oracle's expert-major
one, and by the linearity of the latent up projection."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from synth import quantize_nvfp4


def test_relu2_mlp_hand_example():
    x = np.array([[1.0, 2.0]])
    w_up = np.array([[1.0, -1.0], [2.0, 0.5], [0.0, 1.0]])      # [I=3, d=2]
    w_down = np.array([[1.0, 1.0, 1.0], [0.5, -1.0, 2.0]])      # [d=2, I=3]
    # u = [-1, 3, 2]; relu(u)^2 = [0, 9, 4]; y = [13, -1]
    np.testing.assert_array_equal(O.relu2_mlp(x, w_up, w_down, False), [[13.0, -1.0]])
    np.testing.assert_array_equal(O.relu2_mlp(x, w_up, w_down, True), [[13.0, -1.0]])


def test_relu2_mlp_rounds_at_the_two_bf16_points():
    w_down = np.array([[1.0]])
    # up output 1 + 2^-8 is a BF16 tie: rounds to 1, so relu^2 = 1
    x = np.array([[1.0, 2.0 ** -8]])
    w_up = np.array([[1.0, 1.0]])
    assert O.relu2_mlp(x, w_up, w_down, True)[0, 0] == 1.0
    assert O.relu2_mlp(x, w_up, w_down, False)[0, 0] == (1.0 + 2.0 ** -8) ** 2
    # up output 1 + 2^-7 is exact; its square 1 + 2^-6 + 2^-14 rounds to 1 + 2^-6
    x2 = np.array([[1.0 + 2.0 ** -7]])
    assert O.relu2_mlp(x2, np.array([[1.0]]), w_down, True)[0, 0] == 1.0 + 2.0 ** -6


def _rand_weights(rng, E, d, I, S, L=0):
    w = {"w_router": rng.standard_normal((E, d)).astype(np.float32) / np.sqrt(d),
         "bias": rng.uniform(-0.1, 0.1, E).astype(np.float32)}
    de = L if L else d
    if L:
        w["w_lat_down"] = rng.standard_normal((L, d)) / np.sqrt(d)
        w["w_lat_up"] = rng.standard_normal((d, L)) / np.sqrt(L)
    w["w_up"] = rng.standard_normal((E, I, de)) / np.sqrt(de)
    w["w_down"] = rng.standard_normal((E, de, I)) / np.sqrt(I)
    if S:
        w["w_sh_up"] = rng.standard_normal((S, d)) / np.sqrt(d)
        w["w_sh_down"] = rng.standard_normal((d, S)) / np.sqrt(S)
    return w


def test_one_expert_top1_layer_is_a_scaled_dense_mlp():
    rng = np.random.default_rng(0)
    w = _rand_weights(rng, 1, 32, 24, 0)
    x = rng.standard_normal((9, 32))
    out = O.full_layer(x, w, 1, 1, 1, 1, 1, 2.5, bf16_points=False)
    assert np.all(out["ids"] == 0)
    assert np.all(out["w"] == 2.5)
    dense = O.relu2_mlp(x, w["w_up"][0], w["w_down"][0], False)
    np.testing.assert_allclose(out["y"], 2.5 * dense, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("latent", [0, 12])
@pytest.mark.parametrize("bf16_points", [False, True])
def test_expert_major_layer_equals_token_major_schedule(latent, bf16_points):
    rng = np.random.default_rng(1 + latent)
    E, d, I, S, K = 16, 40, 24, 32, 3
    w = _rand_weights(rng, E, d, I, S, latent)
    x = rng.standard_normal((11, d))
    out = O.full_layer(x, w, E, K, 4, 2, 1, 2.5, bf16_points=bf16_points)
    ids, gw = out["ids"], out["w"]
    # token-major: each token runs its chosen experts, in ascending expert id
    y = np.zeros_like(out["y"])
    for t in range(x.shape[0]):
        xe = x[t:t + 1] @ w["w_lat_down"].T if latent else x[t:t + 1]
        if latent and bf16_points:
            xe = O.bf16_round(xe)
        acc = np.zeros((1, xe.shape[1]))
        for k in np.argsort(ids[t]):
            e = ids[t, k]
            acc += gw[t, k] * O.relu2_mlp(xe, w["w_up"][e], w["w_down"][e], bf16_points)
        if latent:
            acc = (O.bf16_round(acc) if bf16_points else acc) @ w["w_lat_up"].T
        y[t] = acc[0] + O.relu2_mlp(x[t:t + 1], w["w_sh_up"], w["w_sh_down"], bf16_points)[0]
    np.testing.assert_allclose(out["y"], y, rtol=1e-12, atol=1e-12)


def test_latent_up_is_linear_over_the_expert_sum():
    rng = np.random.default_rng(3)
    E, d, L, I, K = 8, 32, 16, 20, 2
    w = _rand_weights(rng, E, d, I, 0, L)
    x = rng.standard_normal((5, d))
    out = O.full_layer(x, w, E, K, 1, 1, 1, 2.5, bf16_points=False)
    xl = x @ w["w_lat_down"].T
    per_expert = np.zeros((5, d))
    for t in range(5):
        for k in range(K):
            e = out["ids"][t, k]
            u = O.relu2_mlp(xl[t:t + 1], w["w_up"][e], w["w_down"][e], False)
            per_expert[t] += out["w"][t, k] * (u @ w["w_lat_up"].T)[0]
    np.testing.assert_allclose(out["y"], per_expert, rtol=1e-12, atol=1e-12)


def test_nvfp4_layer_uses_the_dequantised_experts():
    rng = np.random.default_rng(4)
    E, d, I, K = 4, 32, 32, 2
    w = _rand_weights(rng, E, d, I, 0)
    q = {}
    for name in ("w_up", "w_down"):
        t = torch.from_numpy(w[name].astype(np.float32)).to(torch.bfloat16)
        qq, sf, gs = quantize_nvfp4(t)
        q[name + "_q"], q[name + "_sf"], q[name + "_gs"] = qq.numpy(), sf.numpy(), gs.numpy()
    wq = {k: v for k, v in w.items() if k not in ("w_up", "w_down")}
    wq.update(q)
    deq = dict(w)
    deq["w_up"] = O.dequant_nvfp4(q["w_up_q"], q["w_up_sf"], q["w_up_gs"])
    deq["w_down"] = O.dequant_nvfp4(q["w_down_q"], q["w_down_sf"], q["w_down_gs"])
    x = rng.standard_normal((6, d))
    a = O.full_layer(x, wq, E, K, 1, 1, 1, 5.0, bf16_points=True)
    b = O.full_layer(x, deq, E, K, 1, 1, 1, 5.0, bf16_points=True)
    np.testing.assert_array_equal(a["y"], b["y"])
    # and the dequantised experts are close to the BF16 originals
    assert np.abs(deq["w_up"] - w["w_up"]).max() < 0.25 * np.abs(w["w_up"]).max()


def test_logit_scale_bounds_the_summation_error():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((8, 2688)).astype(np.float32).astype(np.float64)
    wr = (rng.standard_normal((128, 2688)) / 52).astype(np.float32)
    z, scale = O.router_logits(x, wr)
    z32 = (x.astype(np.float32) @ wr.T.astype(np.float32)).astype(np.float64)   # another order, FP32
    assert np.all(np.abs(z32 - z) <= 1e-5 * scale)

"""Pins for the oracle's backward (page "M6.1 Routed Capacity", section 0x06F).

The pages derive the backward of a softmax-gated SwiGLU layer and check it by
central differences with the selected ids frozen (section 0x06F.8).  This
layer's gate (sigmoid, normalise, scale) and experts (ReLU^2) differ, so the
oracle's backward is pinned the same way: every gradient against central
differences of the oracle's own forward (a separate code path) at a point
whose selection does not change under the perturbations, plus the
normalisation identity, the sparsity of the expert and router gradients and
linearity in the upstream gradient."""
import numpy as np
import pytest

from oracle import moe_oracle as O

E, K, G, TG, D_MODEL, L, I, S, T = 8, 2, 2, 1, 12, 8, 10, 14, 3
RSF = 2.5


def _weights(rng, latent):
    de = L if latent else D_MODEL
    w = {"w_router": rng.standard_normal((E, D_MODEL)) / np.sqrt(D_MODEL),
         "bias": rng.uniform(-0.1, 0.1, E),
         "w_up": rng.standard_normal((E, I, de)) / np.sqrt(de),
         "w_down": rng.standard_normal((E, de, I)) / np.sqrt(I),
         "w_sh_up": rng.standard_normal((S, D_MODEL)) / np.sqrt(D_MODEL),
         "w_sh_down": rng.standard_normal((D_MODEL, S)) / np.sqrt(S)}
    if latent:
        w["w_lat_down"] = rng.standard_normal((L, D_MODEL)) / np.sqrt(D_MODEL)
        w["w_lat_up"] = rng.standard_normal((D_MODEL, L)) / np.sqrt(L)
    return w


def _scores(x, w):
    z = x @ w["w_router"].T
    return 1.0 / (1.0 + np.exp(-z))


def _route(x, w, norm):
    s = _scores(x, w)
    ids, _ = O.route(s.astype(np.float32), w["bias"].astype(np.float32), G, TG, K, norm, RSF)
    return ids


def _loss(x, w, ids, D, norm):
    """<D, y> with the given ids, gates from float64 sigmoid scores."""
    s = np.take_along_axis(_scores(x, w), ids.astype(np.int64), axis=1)
    g = RSF * (s / s.sum(axis=1, keepdims=True) if norm else s)
    y = O.layer_forward(x, w, ids, g, E, bf16_points=False)["y"]
    return float(np.sum(D * y))


def _fd(f, arr, idx, h=1e-5):
    old = arr[idx]
    arr[idx] = old + h
    fp = f()
    arr[idx] = old - h
    fm = f()
    arr[idx] = old
    return (fp - fm) / (2 * h)


@pytest.mark.parametrize("latent", [False, True])
@pytest.mark.parametrize("norm", [1, 0])
def test_layer_backward_matches_central_differences(latent, norm):
    rng = np.random.default_rng(100 + latent * 2 + norm)
    w = _weights(rng, latent)
    x = rng.standard_normal((T, D_MODEL))
    D = rng.standard_normal((T, D_MODEL))
    ids = _route(x, w, norm)
    g = O.layer_backward(x, w, ids, _scores(x, w), D, E, norm, RSF)

    def check(name, arr, grad, coords):
        for idx in coords:
            num = _fd(lambda: _loss(x, w, ids, D, norm), arr, idx)
            assert np.array_equal(_route(x, w, norm), ids)
            ana = grad[idx]
            assert abs(ana - num) <= 1e-7 + 1e-6 * abs(ana), f"{name}{idx}: {ana} vs {num}"

    check("dx", x, g["dx"], [(t, j) for t in range(T) for j in range(D_MODEL)])
    pick = lambda shape, n: [tuple(int(rng.integers(0, m)) for m in shape) for _ in range(n)]
    sel = sorted(set(ids.reshape(-1).tolist()))
    check("d_w_router", w["w_router"], g["d_w_router"], [(e, j) for e in sel for j in (0, 5, 11)])
    for e in sel:
        check(f"d_w_up[{e}]", w["w_up"][e], g["d_w_up"][e], pick(w["w_up"][e].shape, 4))
        check(f"d_w_down[{e}]", w["w_down"][e], g["d_w_down"][e], pick(w["w_down"][e].shape, 4))
    check("d_w_sh_up", w["w_sh_up"], g["d_w_sh_up"], pick(w["w_sh_up"].shape, 6))
    check("d_w_sh_down", w["w_sh_down"], g["d_w_sh_down"], pick(w["w_sh_down"].shape, 6))
    if latent:
        check("d_w_lat_down", w["w_lat_down"], g["d_w_lat_down"], pick(w["w_lat_down"].shape, 6))
        check("d_w_lat_up", w["w_lat_up"], g["d_w_lat_up"], pick(w["w_lat_up"].shape, 6))


def test_unchosen_experts_get_no_gradient_and_normalisation_is_scale_free():
    rng = np.random.default_rng(7)
    w = _weights(rng, False)
    x = rng.standard_normal((T, D_MODEL))
    D = rng.standard_normal((T, D_MODEL))
    ids = _route(x, w, 1)
    s = _scores(x, w)
    g = O.layer_backward(x, w, ids, s, D, E, 1, RSF)
    sel = set(ids.reshape(-1).tolist())
    assert set(g["d_w_up"]) == sel and set(g["d_w_down"]) == sel
    for e in range(E):
        if e not in sel:
            assert np.all(g["d_w_router"][e] == 0.0)
    # w is unchanged when every chosen score is scaled by one factor, so the
    # score gradient is orthogonal to the chosen scores
    s_sel = np.take_along_axis(s, ids.astype(np.int64), axis=1)
    np.testing.assert_allclose(np.sum(g["ds"] * s_sel, axis=1), 0.0, atol=1e-12)
    # without normalisation the weights are rsf * s: ds = rsf * q
    g0 = O.layer_backward(x, w, ids, s, D, E, 0, RSF)
    np.testing.assert_allclose(g0["ds"], RSF * g0["q"], rtol=1e-14)


def test_backward_is_linear_in_the_upstream_gradient():
    rng = np.random.default_rng(8)
    w = _weights(rng, True)
    x = rng.standard_normal((T, D_MODEL))
    D1, D2 = rng.standard_normal((2, T, D_MODEL))
    ids = _route(x, w, 1)
    s = _scores(x, w)
    g1 = O.layer_backward(x, w, ids, s, D1, E, 1, RSF)
    g2 = O.layer_backward(x, w, ids, s, D2, E, 1, RSF)
    g3 = O.layer_backward(x, w, ids, s, 2.0 * D1 - D2, E, 1, RSF)
    np.testing.assert_allclose(g3["dx"], 2.0 * g1["dx"] - g2["dx"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g3["d_w_router"], 2.0 * g1["d_w_router"] - g2["d_w_router"], atol=1e-12)


def test_block_backward_matches_central_differences():
    rng = np.random.default_rng(9)
    w = _weights(rng, False)
    x = rng.standard_normal((T, D_MODEL)) * 1.7
    gamma = rng.uniform(0.5, 1.5, D_MODEL)
    eps = 1e-3
    D = rng.standard_normal((T, D_MODEL))
    xn = O.rms_norm(x, gamma, eps)
    ids = _route(xn, w, 1)

    def loss():
        xn_ = O.rms_norm(x, gamma, eps)
        s = np.take_along_axis(_scores(xn_, w), ids.astype(np.int64), axis=1)
        g = RSF * s / s.sum(axis=1, keepdims=True)
        out = O.block_forward(x, gamma, eps, w, ids, g, E, bf16_points=False)["out"]
        return float(np.sum(D * out))

    g = O.block_backward(x, gamma, eps, w, ids, _scores(xn, w), D, E, 1, RSF)
    for idx in [(t, j) for t in range(T) for j in range(D_MODEL)]:
        num = _fd(loss, x, idx)
        assert abs(g["dx"][idx] - num) <= 1e-7 + 1e-6 * abs(num), (idx, g["dx"][idx], num)
    for j in range(D_MODEL):
        num = _fd(loss, gamma, j)
        assert abs(g["d_norm_w"][j] - num) <= 1e-7 + 1e-6 * abs(num), (j, g["d_norm_w"][j], num)


def test_bf16_points_change_nothing_when_every_operand_is_representable():
    # small integers and powers of two: a, h, dU, dh, da and all products are
    # exact in BF16, so the rounding points must leave every gradient unchanged
    rng = np.random.default_rng(11)
    d, E_, I_ = 8, 4, 8
    w = {"w_router": rng.integers(-2, 3, (E_, d)).astype(np.float64) / 8,
         "w_up": rng.integers(-2, 3, (E_, I_, d)).astype(np.float64) / 4,
         "w_down": rng.integers(-2, 3, (E_, d, I_)).astype(np.float64) / 4}
    x = rng.integers(-2, 3, (3, d)).astype(np.float64)
    D = rng.integers(-2, 3, (3, d)).astype(np.float64)
    ids = np.array([[0, 2], [1, 3], [2, 0]])
    scores = np.full((3, E_), 0.5)
    a = O.layer_backward(x, w, ids, scores, D, E_, 0, 1.0, bf16_points=False)
    b = O.layer_backward(x, w, ids, scores, D, E_, 0, 1.0, bf16_points=True)
    for k in ("dx", "d_w_router"):
        np.testing.assert_array_equal(a[k], b[k])
    for e in a["d_w_up"]:
        np.testing.assert_array_equal(a["d_w_up"][e], b["d_w_up"][e])
        np.testing.assert_array_equal(a["d_w_down"][e], b["d_w_down"][e])


def test_bf16_points_round_the_backward_operands():
    # a gate of 1/3 makes dU = w dy inexact in BF16: the rounded run differs,
    # by at most one BF16 step of dU, where dU enters
    rng = np.random.default_rng(12)
    d, E_, I_ = 8, 2, 8
    w = {"w_router": rng.standard_normal((E_, d)), "w_up": np.ones((E_, I_, d)) / 8,
         "w_down": np.ones((E_, d, I_)) / 8}
    x = np.ones((1, d))
    D = np.ones((1, d))
    ids = np.array([[0]])
    scores = np.array([[1.0 / 3.0, 0.5]])
    a = O.layer_backward(x, w, ids, scores, D, E_, 0, 1.0, bf16_points=False)
    b = O.layer_backward(x, w, ids, scores, D, E_, 0, 1.0, bf16_points=True)
    rel = np.abs(b["d_w_down"][0] - a["d_w_down"][0]) / np.abs(a["d_w_down"][0])
    assert 0 < rel.max() <= 2.0 ** -8

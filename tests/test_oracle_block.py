"""Pins for the oracle's RMSNorm and MoE block (page "Nemotron Is Not One
Circuit", section "The Four Layer Kinds CKE Must Preserve": an MoE layer is
RMSNorm -> router -> group-limited top-k -> routed ReLU^2 experts + shared
expert -> residual).

The pages name RMSNorm without a formula; these pins fix the reading the
oracle takes (root mean square over the hidden width, no mean subtraction, a
per-column weight, epsilon inside the root) by hand-computed values and closed
forms, and pin the block by the residual identity and a one-expert dense
evaluation written out here."""
import numpy as np

from oracle import moe_oracle as O


def test_rms_norm_hand_example():
    # x = [3, 4]: mean square 12.5, root 3.5355339059327378
    x = np.array([[3.0, 4.0]])
    got = O.rms_norm(x, np.ones(2), 0.0)
    np.testing.assert_allclose(got, [[0.8485281374238571, 1.1313708498984762]], rtol=1e-15)
    # gamma scales each column; eps enters inside the root: 12.5 + 3.5 = 16, root 4
    got = O.rms_norm(x, np.array([2.0, 0.5]), 3.5)
    np.testing.assert_array_equal(got, [[1.5, 0.5]])


def test_rms_norm_of_a_constant_row_is_its_sign():
    x = np.array([[-2.5] * 8, [7.0] * 8])
    np.testing.assert_allclose(O.rms_norm(x, np.ones(8), 0.0), [[-1.0] * 8, [1.0] * 8], rtol=1e-15)


def test_rms_norm_mean_square_closed_form():
    # mean((xn / gamma)^2) = ms / (ms + eps): a dropped square, a sum in place of
    # the mean or eps outside the root all break it
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 64)) * 3.0
    gamma = rng.uniform(0.5, 1.5, 64)
    eps = 0.25
    xn = O.rms_norm(x, gamma, eps)
    ms = np.mean(x * x, axis=1)
    np.testing.assert_allclose(np.mean((xn / gamma) ** 2, axis=1), ms / (ms + eps), rtol=1e-13)


def test_rms_norm_is_scale_invariant_without_eps_and_not_with_it():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 32))
    g = rng.uniform(0.5, 1.5, 32)
    np.testing.assert_allclose(O.rms_norm(37.0 * x, g, 0.0), O.rms_norm(x, g, 0.0), rtol=1e-13)
    assert not np.allclose(O.rms_norm(0.01 * x, g, 1e-2), O.rms_norm(x, g, 1e-2), rtol=1e-3)


def _weights(rng, E, d, I, S, L=0):
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


def test_block_with_silent_outputs_is_the_identity():
    # zero down projections (routed and shared) and a zero latent up: out = x exactly
    rng = np.random.default_rng(5)
    for L in (0, 16):
        w = _weights(rng, 4, 32, 24, 40, L)
        w["w_down"] = np.zeros_like(w["w_down"])
        w["w_sh_down"] = np.zeros_like(w["w_sh_down"])
        if L:
            w["w_lat_up"] = np.zeros_like(w["w_lat_up"])
        x = rng.standard_normal((6, 32))
        ids = np.array([[0, 2]] * 6)
        gw = np.full((6, 2), 1.25)
        out = O.block_forward(x, np.ones(32), 1e-5, w, ids, gw, 4, bf16_points=False)
        np.testing.assert_array_equal(out["out"], x)


def test_one_expert_block_against_a_dense_evaluation():
    # E = 1, K = 1: out = x + w * W_down relu(W_up xn)^2 + W_sd relu(W_su xn)^2,
    # xn = gamma * x / sqrt(mean(x^2) + eps), all written out here
    rng = np.random.default_rng(6)
    d, I, S = 16, 12, 20
    w = _weights(rng, 1, d, I, S)
    x = rng.standard_normal((4, d)) * 2.0
    gamma = rng.uniform(0.5, 1.5, d)
    eps = 1e-3
    out = O.block_forward(x, gamma, eps, w, np.zeros((4, 1), dtype=np.int64), np.full((4, 1), 2.5), 1,
                          bf16_points=False)
    for t in range(4):
        r = 1.0 / np.sqrt(np.sum(x[t] ** 2) / d + eps)
        xn = gamma * x[t] * r
        routed = 2.5 * w["w_down"][0] @ np.maximum(w["w_up"][0] @ xn, 0.0) ** 2
        shared = w["w_sh_down"] @ np.maximum(w["w_sh_up"] @ xn, 0.0) ** 2
        np.testing.assert_allclose(out["out"][t], x[t] + routed + shared, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(out["xn_ref"][t], xn, rtol=1e-14)


def test_block_reads_the_given_normalised_rows():
    # with xn given, the layer part sees exactly those rows (the device's stored
    # rows); out still adds the unnormalised residual x
    rng = np.random.default_rng(7)
    w = _weights(rng, 2, 16, 8, 0)
    x = rng.standard_normal((3, 16))
    xn = rng.standard_normal((3, 16))
    ids = np.array([[1], [0], [1]])
    gw = np.ones((3, 1))
    out = O.block_forward(x, np.ones(16), 0.0, w, ids, gw, 2, bf16_points=False, xn=xn)
    for t in range(3):
        e = ids[t, 0]
        y = w["w_down"][e] @ np.maximum(w["w_up"][e] @ xn[t], 0.0) ** 2
        np.testing.assert_allclose(out["out"][t], x[t] + y, rtol=1e-12, atol=1e-12)

"""GPU parity of the ReLU^2-sparse down projection (page "Nemotron-3.5-Super
120B on an 8 GB GPU", section "The engine, step by step", item 4 "Skip the
zeros"): the group-major re-layout is the documented byte permutation of
W_down, and a decode layer given the re-laid weights matches the oracle (which
never skips) on inputs with the page's ReLU^2 sparsity, on plain random inputs
(nothing to skip) and on inputs where whole experts are dead."""
import numpy as np
import pytest
import torch

from synth import (BF16, NANO_DECODE, NANO_DECODE_SPARSE, SUPER_LATENT, SUPER_NVFP4_SPARSE, make_x, scaled)

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import routed_relu_expert_gb300 as M
    from routed_relu_expert_gb300 import _native as N
    from gpu_helpers import (check_output, check_route_tables, check_router, device_weights, oracle_weights, to_np,
                             tol_of, ws_table)

SMALL_BF16 = scaled(NANO_DECODE, name="sparse_small_bf16", d_model=512, n_experts=16, top_k=4, d_expert=320,
                    d_shared=384, weight_seed=43, tokens=())
SMALL_BF16_SPARSE = scaled(SMALL_BF16, name="sparse_small_bf16_s", relu_sparsity=0.925)
SMALL_BF16_DEAD = scaled(SMALL_BF16, name="sparse_small_bf16_dead", relu_sparsity=0.9995)
SMALL_NVFP4_SPARSE = scaled(SUPER_LATENT, name="sparse_small_nvfp4_s", d_model=512, d_latent=256, n_experts=64,
                            top_k=6, n_group=8, topk_group=4, d_expert=384, d_shared=448, expert_dtype=2,
                            relu_sparsity=0.925, weight_seed=47, tokens=())


def _expected_layout(shape, w):
    """The group-major layout as the header defines it, built on the host."""
    E, de, I = shape.n_experts, shape.d_e, shape.d_expert
    if shape.expert_dtype != 2:
        W = w["w_down"].view(torch.int16).cpu().numpy().reshape(E, de, I)
        # [E, g, o, l, 8]: lane l = 4r + t -> rows 16o + r and 16o + r + 8, neurons 16g + 4t .. +3
        blk = W.reshape(E, de // 16, 2, 8, I // 16, 4, 4)            # e, o, half, r, g, t, k
        out = blk.transpose(0, 4, 1, 3, 5, 2, 6)                      # e, g, o, r, t, half, k
        return out.reshape(-1).view(np.uint8), None
    q = w["w_down_q"].cpu().numpy().reshape(E, de, I // 2)
    sf = w["w_down_sf"].cpu().numpy().reshape(E, de, I // 16)
    # values [E, g, quad, l, tile j, half, 2 bytes]: bytes 8g + 2t, +1 of row 64 quad + 16 j + r + 8 half
    v = q.reshape(E, de // 64, 4, 2, 8, I // 16, 4, 2)               # e, quad, j, half, r, g, t, byte
    vo = v.transpose(0, 5, 1, 4, 6, 2, 3, 7)                          # e, g, quad, r, t, j, half, byte
    # scales [E, g, quad, r, tile j, half]
    s = sf.reshape(E, de // 64, 4, 2, 8, I // 16)                     # e, quad, j, half, r, g
    so = s.transpose(0, 5, 1, 4, 2, 3)                                # e, g, quad, r, j, half
    return vo.reshape(-1), so.reshape(-1)


@pytest.mark.parametrize("shape", ["bf16", "nvfp4"])
def test_layout_is_the_documented_permutation(shape):
    s = {"bf16": SMALL_BF16, "nvfp4": SMALL_NVFP4_SPARSE}[shape]
    w = device_weights(s)
    layer = M.MoELayer(M.config_from(s), w)
    got = M.sparse_down_layout(layer.cfg, layer.weights)
    torch.cuda.synchronize()
    want_v, want_s = _expected_layout(s, w)
    assert np.array_equal(got["w_down_g"].cpu().numpy(), want_v)
    if want_s is not None:
        assert np.array_equal(got["w_down_g_sf"].cpu().numpy(), want_s)


def _dead_group_fraction(shape, ws, T):
    """Fraction of (expert, 16-neuron group) pairs of the step whose h values
    are zero in every row of the expert (what the sparse kernel skips)."""
    cfg = M.config_from(shape)
    R, I = T * shape.top_k, shape.d_expert
    h = ws_table(ws, cfg, T, N.MOE_WS_H, torch.int16).view(R, I).cpu().numpy() & 0x7FFF
    offs = ws_table(ws, cfg, T, N.MOE_WS_OFFSETS, torch.int32).cpu().numpy()
    dead = tot = 0
    for e in range(shape.n_experts):
        a, b = offs[e], offs[e + 1]
        if b > a:
            live = (h[a:b].reshape(b - a, I // 16, 16) != 0).any(axis=(0, 2))
            dead += int(np.sum(~live))
            tot += live.size
    return dead / tot


def _sparse_parity(shape, T, min_dead=None):
    w = device_weights(shape)
    cfg = M.config_from(shape)
    layer = M.MoELayer(cfg, w)
    layer.enable_sparse_down()
    x = make_x(shape, T, "cuda")
    E, K = shape.n_experts, shape.top_k
    g = {"y": torch.empty_like(x), "ids": torch.empty((T, K), dtype=torch.int32, device="cuda"),
         "topw": torch.empty((T, K), dtype=torch.float32, device="cuda"),
         "logits": torch.empty((T, E), dtype=torch.float32, device="cuda"),
         "scores": torch.empty((T, E), dtype=torch.float32, device="cuda")}
    layer.forward(x, g["y"], ids_out=g["ids"], topw_out=g["topw"], logits_out=g["logits"], scores_out=g["scores"])
    ws = layer.workspace(T, x.device)
    assert M.moe_get_device_error(ws) == 0
    dead = _dead_group_fraction(shape, ws, T)
    if min_dead is not None:
        assert dead >= min_dead, f"only {dead:.3f} of the groups are dead: the input does not exercise skipping"
    # the same layer without the group-major weights: routing identical, output close
    dense = M.MoELayer(cfg, w)
    y_dense = torch.empty_like(x)
    ids_dense = torch.empty_like(g["ids"])
    dense.forward(x, y_dense, ids_out=ids_dense)
    torch.cuda.synchronize()
    assert torch.equal(ids_dense, g["ids"])
    gn = to_np(g)
    check_route_tables(shape, ws, gn["ids"], T)
    ow = oracle_weights(w)
    x_np = x.float().cpu().numpy().astype(np.float64)
    ids_o, w_o = check_router(shape, x_np, ow, gn)
    err = check_output(shape, x_np, ow, ids_o, w_o, gn["y"], tol_of(shape))
    err_dense = check_output(shape, x_np, ow, ids_o, w_o, y_dense.float().cpu().numpy(), tol_of(shape))
    return err, err_dense, dead


@pytest.mark.parametrize("T", [1, 2, 4, 16, 64])
def test_nano_sparse_decode(T):
    # a 16-neuron group of one token is dead with probability near 0.925^16
    _sparse_parity(NANO_DECODE_SPARSE, T, min_dead=0.2 if T == 1 else None)


@pytest.mark.parametrize("T", [1, 2, 9])
def test_super_nvfp4_sparse_decode(T):
    # below 8 tokens the FP16 decode path runs the sparse down product; at 9
    # the FP4 tensor path (the group-major weights are present but unused)
    _sparse_parity(SUPER_NVFP4_SPARSE, T, min_dead=0.2 if T == 1 else None)


@pytest.mark.parametrize("shape,T", [("bf16", 1), ("bf16", 7), ("bf16", 64), ("sparse", 3), ("dead", 1),
                                     ("dead", 5), ("nvfp4", 1)])
def test_scaled_sparse_down(shape, T):
    s = {"bf16": SMALL_BF16, "sparse": SMALL_BF16_SPARSE, "dead": SMALL_BF16_DEAD,
         "nvfp4": SMALL_NVFP4_SPARSE}[shape]
    _, _, dead = _sparse_parity(s, T)
    if shape == "dead":
        assert dead > 0.9


def test_sparse_down_unsupported_configurations_are_refused():
    from synth import TINY_FP32
    cfg = M.config_from(TINY_FP32)
    with pytest.raises(M.MoEError):
        M.sparse_down_bytes(cfg)

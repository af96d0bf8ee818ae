"""GPU parity of the MoE block (out = x + layer(RMSNorm(x))) against the oracle.

Each step is checked on the device's own input to that step, as the layer's
tests do: the normalised rows xn against the oracle's float64 RMSNorm of x
(within one rounding to the activation type); the router, the dispatch tables
and the routed output on the device's xn; the output against
x + oracle layer(xn), within the layer's tolerance times RMS of the layer
output plus the output's own rounding.  Verify shapes T = 1, 2, 4, 8, 16 (page
"NemotronH (Nemotron 3.5 Lightning, Bolt, Super VL)", section "Speculation":
verify blocks of 1 to 16 rows), the tensor-core path above 64 tokens, in-place
use, and a chain of blocks captured in one CUDA graph."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from synth import BF16, F32, NANO_DECODE, SUPER_LATENT, SUPER_NVFP4, TINY_FP32, make_norm_weight, make_x, scaled

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import routed_relu_expert_gb300 as M
    from gpu_helpers import check_route_tables, check_router, device_weights, oracle_weights, to_np, tol_of

EPS = 1e-5

SMALL_NANO = scaled(NANO_DECODE, name="nano_scaled_block", d_model=512, n_experts=32, top_k=4, d_expert=320,
                    d_shared=384, weight_seed=23, tokens=())
SMALL_SUPER = scaled(SUPER_LATENT, name="super_scaled_block", d_model=512, d_latent=256, n_experts=64, top_k=6,
                     n_group=8, topk_group=4, d_expert=320, d_shared=448, weight_seed=29, tokens=())
SMALL_NVFP4 = scaled(SUPER_LATENT, name="nvfp4_scaled_block", d_model=512, d_latent=256, n_experts=64, top_k=6,
                     n_group=8, topk_group=4, d_expert=384, d_shared=448, expert_dtype=2, weight_seed=31,
                     tokens=())
NO_SHARED = scaled(NANO_DECODE, name="nano_no_shared_block", d_model=256, n_experts=16, top_k=2, d_expert=128,
                   d_shared=0, weight_seed=37, tokens=())


def run_block(shape, w, gamma, x, out=None):
    cfg = M.config_from(shape)
    T, E, K = x.shape[0], shape.n_experts, shape.top_k
    blk = M.MoEBlock(cfg, w, gamma, EPS)
    out = torch.empty_like(x) if out is None else out
    xn = torch.empty_like(x)
    ids = torch.empty((T, K), dtype=torch.int32, device="cuda")
    topw = torch.empty((T, K), dtype=torch.float32, device="cuda")
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    scores = torch.empty((T, E), dtype=torch.float32, device="cuda")
    blk.forward(x, out, x_norm_out=xn, ids_out=ids, topw_out=topw, logits_out=logits, scores_out=scores)
    ws = blk.workspace(T, x.device)
    err = M.moe_get_device_error(ws)
    torch.cuda.synchronize()
    return {"y": out, "xn": xn, "ids": ids, "topw": topw, "logits": logits, "scores": scores, "err": err,
            "ws": ws}


def check_xn(shape, x_np, gamma_np, xn_gpu):
    """Device xn against the float64 RMSNorm: one rounding to BF16 (2^-9
    relative) plus FP32 arithmetic for BF16 rows; FP32 rows within 1e-5 of
    the row's largest value."""
    ref = O.rms_norm(x_np, gamma_np, EPS)
    d = np.abs(xn_gpu.astype(np.float64) - ref)
    if shape.act_dtype == BF16:
        bound = 2.0 ** -8 * np.abs(ref) + 1e-30
    else:
        bound = 1e-5 * np.max(np.abs(ref), axis=1, keepdims=True)
    assert np.all(d <= bound), f"xn off by {np.max(d / np.maximum(bound, 1e-30)):.2f} x its bound"


def check_block_output(shape, x_np, ow, xn_gpu, ids_o, w_o, out_gpu):
    """out against x + layer(xn) on the device's xn and routing; the bar is the
    layer's tolerance times RMS of the layer output, plus the output's rounding
    (relative to |out|, which includes the residual)."""
    lay = O.block_forward(x_np, np.ones(x_np.shape[1]), EPS, ow, ids_o, w_o, shape.n_experts,
                          bf16_points=shape.act_dtype == BF16, xn=xn_gpu)
    want = lay["out"]
    rms = float(np.sqrt(np.mean(lay["y"] ** 2)))
    rnd = 2.0 ** -8 if shape.act_dtype == BF16 else 1e-6
    d = np.abs(out_gpu.astype(np.float64) - want)
    excess = d - rnd * np.abs(want)
    err = float(np.max(excess)) / rms
    assert err <= tol_of(shape), f"max |out - ref| beyond rounding = {err:.3e} RMS(layer) > {tol_of(shape)}"
    return err


def block_parity(shape, T, seed_stream=0, replica=0):
    w = device_weights(shape, replica)
    gamma = make_norm_weight(shape, "cuda", replica)
    x = make_x(shape, T, "cuda", seed_stream)
    g = run_block(shape, w, gamma, x)
    assert g["err"] == 0
    ws = g.pop("ws")
    g = to_np(g)
    check_route_tables(shape, ws, g["ids"], T)
    ow = oracle_weights(w)
    x_np = x.float().cpu().numpy().astype(np.float64)
    check_xn(shape, x_np, gamma.cpu().numpy().astype(np.float64), g["xn"])
    xn64 = g["xn"].astype(np.float64)
    ids_o, w_o = check_router(shape, xn64, ow, g)
    return check_block_output(shape, x_np, ow, xn64, ids_o, w_o, g["y"]), x, g


@pytest.mark.parametrize("T", [1, 2, 4, 8, 16])
def test_nano_block_verify_shapes(T):
    block_parity(NANO_DECODE, T)


@pytest.mark.parametrize("T", [1, 2, 8, 16])
def test_super_latent_block_verify_shapes(T):
    block_parity(SUPER_LATENT, T)


@pytest.mark.parametrize("T", [1, 4, 16])
def test_super_nvfp4_block_verify_shapes(T):
    block_parity(SUPER_NVFP4, T)


@pytest.mark.parametrize("T", [1, 16, 100])
def test_fp32_block(T):
    block_parity(TINY_FP32, T)


@pytest.mark.parametrize("shape,T", [("nano", 200), ("super", 200), ("nvfp4", 200), ("nvfp4", 9),
                                     ("no_shared", 5), ("no_shared", 130)])
def test_scaled_blocks_every_path(shape, T):
    # above 64 tokens the output passes through the tensor-core epilogue
    # (latent up) or the combine (no latent); no shared expert: the combine alone
    s = {"nano": SMALL_NANO, "super": SMALL_SUPER, "nvfp4": SMALL_NVFP4, "no_shared": NO_SHARED}[shape]
    block_parity(s, T)


@pytest.mark.parametrize("shape,T", [("nano", 4), ("super", 200)])
def test_block_in_place_is_bit_identical(shape, T):
    s = {"nano": NANO_DECODE, "super": SMALL_SUPER}[shape]
    w = device_weights(s)
    gamma = make_norm_weight(s, "cuda")
    x = make_x(s, T, "cuda")
    ref = run_block(s, w, gamma, x)["y"].clone()
    xi = x.clone()
    got = run_block(s, w, gamma, xi, out=xi)
    assert got["err"] == 0
    assert torch.equal(xi.view(torch.int16), ref.view(torch.int16))


def test_block_rejects_partial_overlap_and_bad_eps():
    s = SMALL_NANO
    cfg = M.config_from(s)
    w = device_weights(s)
    blk = M.MoEBlock(cfg, w, make_norm_weight(s, "cuda"), EPS)
    buf = torch.zeros((9, s.d_model), dtype=torch.bfloat16, device="cuda")
    x = buf[:8]
    with pytest.raises(M.MoEError):
        blk.forward(x, buf[1:9])                      # out overlaps x without being x
    with pytest.raises(M.MoEError):
        blk.forward(x, torch.empty_like(x), x_norm_out=x)
    bad = M.MoEBlock(cfg, w, make_norm_weight(s, "cuda"), -1.0)
    with pytest.raises(M.MoEError):
        bad.forward(x)


@pytest.mark.parametrize("shape,T", [("nano", 4), ("nvfp4", 8)])
def test_chain_of_blocks_in_one_graph(shape, T):
    """Three blocks (independent weights) chained through the residual stream
    and captured in one CUDA graph: the replay reproduces the eager chain bit
    for bit, and each block matches the oracle on its own device input."""
    s = {"nano": NANO_DECODE, "nvfp4": SUPER_NVFP4}[shape]
    n = 3
    cfg = M.config_from(s)
    ws_ = [device_weights(s, r) for r in range(n)]
    gammas = [make_norm_weight(s, "cuda", r) for r in range(n)]
    blocks = [M.MoEBlock(cfg, ws_[r], gammas[r], EPS) for r in range(n)]
    x0 = make_x(s, T, "cuda", 5)
    bufs = [torch.empty_like(x0) for _ in range(n)]
    ids = [torch.empty((T, s.top_k), dtype=torch.int32, device="cuda") for _ in range(n)]
    topw = [torch.empty((T, s.top_k), dtype=torch.float32, device="cuda") for _ in range(n)]
    logits = [torch.empty((T, s.n_experts), dtype=torch.float32, device="cuda") for _ in range(n)]
    scores = [torch.empty((T, s.n_experts), dtype=torch.float32, device="cuda") for _ in range(n)]
    xns = [torch.empty_like(x0) for _ in range(n)]
    ws = M.new_workspace(cfg, T)
    for b in blocks:
        b._ws = ws

    def chain():
        cur = x0
        for r in range(n):
            blocks[r].forward(cur, bufs[r], x_norm_out=xns[r], ids_out=ids[r], topw_out=topw[r],
                              logits_out=logits[r], scores_out=scores[r])
            cur = bufs[r]

    chain()
    torch.cuda.synchronize()
    eager = [b.clone() for b in bufs]
    for b in bufs:
        b.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chain()
    g.replay()
    torch.cuda.synchronize()
    assert M.moe_get_device_error(ws) == 0
    for r in range(n):
        assert torch.equal(bufs[r].view(torch.int16), eager[r].view(torch.int16)), f"block {r} replay differs"
    cur = x0
    for r in range(n):
        ow = oracle_weights(ws_[r])
        x_np = cur.float().cpu().numpy().astype(np.float64)
        check_xn(s, x_np, gammas[r].cpu().numpy().astype(np.float64), xns[r].float().cpu().numpy())
        xn64 = xns[r].float().cpu().numpy().astype(np.float64)
        gr = to_np({"logits": logits[r], "scores": scores[r], "ids": ids[r], "topw": topw[r]})
        ids_o, w_o = check_router(s, xn64, ow, gr)
        check_block_output(s, x_np, ow, xn64, ids_o, w_o, bufs[r].float().cpu().numpy())
        cur = bufs[r]

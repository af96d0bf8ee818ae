"""GPU parity of the backward (page "M6.1 Routed Capacity", section 0x06F)
against the oracle's float64 backward of the same forward relation.

The device forward runs first and leaves its state in the workspace; the
backward then gets the forward's own ids, weights and scores, so the oracle
differentiates exactly the relation the device froze.  Every gradient is
compared element by element, as |g - g_ref| / (|g_ref| + RMS(g_ref)), with
two references:
 - the oracle with the rounding points (the forward's BF16 points and the
   backward's BF16 operands dU, da, dy_r and the latent input gradient):
   within 5e-2: an operand that rounds the other way at a BF16 boundary
   shifts its term by one BF16 step (2^-8), and the heavy-tailed terms of an
   expert's few rows reach 8-12 x (|g_ref| + RMS) (3.3e-2 measured at worst
   over these cases); the step-by-step test below is the exact check;
 - the exact float64 backward: within 0.15.  The expert weight gradients of a
   few tokens are sums of outer products of heavy-tailed vectors (h is a
   square), so one BF16 rounding of a large term is a large share of a small
   sum; this bar bounds the design's whole error, the first one its
   arithmetic.
Step by step, each weight gradient is also checked on the device's own BF16
operands (read back from the backward scratch) to FP32 accuracy, and each
operand against the oracle's rounding of the device's inputs to within one
BF16 step.  Also: expert and router rows of experts without routes stay
untouched, gradients accumulate, and two runs give the same bits."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from synth import NANO_DECODE, NANO_PREFILL, SUPER_LATENT, make_norm_weight, make_x, scaled

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import routed_relu_expert_gb300 as M
    from gpu_helpers import device_weights, oracle_weights

TOL_GRAD = 5e-2      # against the oracle with the rounding points
TOL_EXACT = 0.15     # against the exact float64 backward
EPS = 1e-5

SMALL_NANO = scaled(NANO_DECODE, name="bwd_nano", d_model=512, n_experts=32, top_k=4, d_expert=320, d_shared=384,
                    weight_seed=53, tokens=())
SMALL_SUPER = scaled(SUPER_LATENT, name="bwd_super", d_model=512, d_latent=256, n_experts=64, top_k=6, n_group=8,
                     topk_group=4, d_expert=320, d_shared=448, weight_seed=59, tokens=())
NO_SHARED = scaled(NANO_DECODE, name="bwd_no_shared", d_model=256, n_experts=16, top_k=2, d_expert=128, d_shared=0,
                   weight_seed=61, tokens=())


def _dy(shape, T, seed=0):
    g = torch.Generator(device="cuda")
    g.manual_seed(1000 + 7 * T + seed)
    return torch.randn((T, shape.d_model), generator=g, device="cuda").to(torch.bfloat16)


def _zero_grads(shape, block=False):
    E, d, L, I, S, de = shape.n_experts, shape.d_model, shape.d_latent, shape.d_expert, shape.d_shared, shape.d_e
    z = lambda *sh: torch.zeros(sh, dtype=torch.float32, device="cuda")
    g = {"d_router": z(E, d), "d_up": z(E, I, de), "d_down": z(E, de, I)}
    if L:
        g["d_lat_down"], g["d_lat_up"] = z(L, d), z(d, L)
    if S:
        g["d_sh_up"], g["d_sh_down"] = z(S, d), z(d, S)
    if block:
        g["d_norm_w"] = z(d)
    return g


def _forward(shape, w, x, gamma=None):
    cfg = M.config_from(shape)
    T, E, K = x.shape[0], shape.n_experts, shape.top_k
    layer = M.MoEBlock(cfg, w, gamma, EPS) if gamma is not None else M.MoELayer(cfg, w)
    st = {"ids": torch.empty((T, K), dtype=torch.int32, device="cuda"),
          "topw": torch.empty((T, K), dtype=torch.float32, device="cuda"),
          "scores": torch.empty((T, E), dtype=torch.float32, device="cuda"),
          "y": torch.empty_like(x)}
    extra = {}
    if gamma is not None:
        st["xn"] = torch.empty_like(x)
        extra["x_norm_out"] = st["xn"]
    layer.forward(x, st["y"], ids_out=st["ids"], topw_out=st["topw"], scores_out=st["scores"], **extra)
    st["ws"] = layer.workspace(T, x.device)
    st["layer"] = layer
    return st


def _compare(name, got, ref, tol=TOL_GRAD, tag="rp"):
    """max over elements of |g - g_ref| / (|g_ref| + RMS(g_ref)): a relative
    error where the gradient is large, an absolute one (against the tensor's
    RMS) where it is small"""
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = float(np.max(np.abs(got.astype(np.float64) - ref) / (np.abs(ref) + max(rms, 1e-30))))
    print(f"GRADERR {tag} {name} {err:.3e}")
    assert err <= tol, f"{name} ({tag}): max |g - g_ref| / (|g_ref| + RMS) = {err:.3e} > {tol}"
    return err


def _check_grads(shape, grads, ref, ids_np, tol=TOL_GRAD, tag="rp", host=None):
    errs = {}
    host = host or {k: v.cpu().numpy() for k, v in grads.items()}
    sel = sorted(set(ids_np.reshape(-1).tolist()))
    un = [e for e in range(shape.n_experts) if e not in sel]
    for e in sel:
        errs[f"d_up[{e}]"] = _compare(f"d_up[{e}]", host["d_up"][e], ref["d_w_up"][e], tol, tag)
        errs[f"d_down[{e}]"] = _compare(f"d_down[{e}]", host["d_down"][e], ref["d_w_down"][e], tol, tag)
    if un:
        idx = torch.tensor(un, device="cuda")
        for k in ("d_up", "d_down", "d_router"):
            assert torch.count_nonzero(grads[k][idx]) == 0, f"{k} touched an expert without routes"
    errs["d_router"] = _compare("d_router", host["d_router"][sel], ref["d_w_router"][sel], tol, tag)
    for k, rk in (("d_sh_up", "d_w_sh_up"), ("d_sh_down", "d_w_sh_down"), ("d_lat_down", "d_w_lat_down"),
                  ("d_lat_up", "d_w_lat_up")):
        if k in grads:
            errs[k] = _compare(k, host[k], ref[rk], tol, tag)
    return errs


def layer_backward_parity(shape, T):
    w = device_weights(shape)
    cfg = M.config_from(shape)
    x = make_x(shape, T, "cuda")
    st = _forward(shape, w, x)
    dy = _dy(shape, T)
    dx = torch.empty((T, shape.d_model), dtype=torch.float32, device="cuda")
    grads = _zero_grads(shape)
    bws = M.new_backward_workspace(cfg, T)
    M.moe_layer_backward(cfg, x, st["layer"].weights, dy, st["ids"], st["topw"], st["scores"], dx, grads,
                         st["ws"], bws)
    assert M.moe_get_device_error(st["ws"]) == 0
    torch.cuda.synchronize()
    ow = oracle_weights(w)
    ids_np = st["ids"].cpu().numpy()
    host = {k: v.cpu().numpy() for k, v in grads.items()}
    errs = {}
    for bp, tol, tag in ((True, TOL_GRAD, "rp"), (False, TOL_EXACT, "exact")):
        ref = O.layer_backward(x.float().cpu().numpy(), ow, ids_np, st["scores"].cpu().numpy(),
                               dy.float().cpu().numpy(), shape.n_experts, shape.norm_topk_prob,
                               shape.routed_scaling_factor, bf16_points=bp)
        errs[tag] = _check_grads(shape, grads, ref, ids_np, tol, tag, host)
        errs[tag]["dx"] = _compare("dx", dx.cpu().numpy(), ref["dx"], tol, tag)
    return errs, (st, dy, dx, grads, bws, x)


@pytest.mark.parametrize("shape,T", [("nano", 1), ("nano", 5), ("nano", 64), ("nano", 200), ("super", 1),
                                     ("super", 13), ("super", 200), ("no_shared", 3), ("no_shared", 130)])
def test_layer_backward_scaled(shape, T):
    s = {"nano": SMALL_NANO, "super": SMALL_SUPER, "no_shared": NO_SHARED}[shape]
    layer_backward_parity(s, T)


@pytest.mark.parametrize("shape,T", [("nano_decode", 4), ("super_latent", 2), ("nano_prefill", 256)])
def test_layer_backward_full_size(shape, T):
    s = {"nano_decode": NANO_DECODE, "super_latent": SUPER_LATENT, "nano_prefill": NANO_PREFILL}[shape]
    layer_backward_parity(s, T)


def test_backward_accumulates_and_is_deterministic():
    s = SMALL_SUPER
    cfg = M.config_from(s)
    _, (st, dy, dx, grads, bws, x) = layer_backward_parity(s, 37)
    first = {k: v.clone() for k, v in grads.items()}
    dx1 = dx.clone()
    M.moe_layer_backward(cfg, x, st["layer"].weights, dy, st["ids"], st["topw"], st["scores"], dx, grads,
                         st["ws"], bws)
    torch.cuda.synchronize()
    assert torch.equal(dx, dx1)
    for k in grads:
        assert torch.equal(grads[k], 2.0 * first[k]), f"{k} did not accumulate exactly"


@pytest.mark.parametrize("shape,T", [("nano_decode", 4), ("super", 9), ("super", 150)])
def test_block_backward(shape, T):
    s = {"nano_decode": NANO_DECODE, "super": SMALL_SUPER}[shape]
    w = device_weights(s)
    cfg = M.config_from(s)
    gamma = make_norm_weight(s, "cuda")
    x = make_x(s, T, "cuda")
    st = _forward(s, w, x, gamma)
    dout = _dy(s, T, 1)
    dx = torch.empty((T, s.d_model), dtype=torch.float32, device="cuda")
    grads = _zero_grads(s, block=True)
    bws = M.new_backward_workspace(cfg, T)
    M.moe_block_backward(cfg, x, gamma, EPS, st["layer"].weights, dout, st["ids"], st["topw"], st["scores"], dx,
                         grads, st["ws"], bws, x_norm=st["xn"])
    torch.cuda.synchronize()
    ow = oracle_weights(w)
    ids_np = st["ids"].cpu().numpy()
    host = {k: v.cpu().numpy() for k, v in grads.items()}
    for bp, tol, tag in ((True, TOL_GRAD, "rp"), (False, TOL_EXACT, "exact")):
        ref = O.block_backward(x.float().cpu().numpy(), gamma.cpu().numpy(), EPS, ow, ids_np,
                               st["scores"].cpu().numpy(), dout.float().cpu().numpy(), s.n_experts,
                               s.norm_topk_prob, s.routed_scaling_factor, xn=st["xn"].float().cpu().numpy(),
                               bf16_points=bp)
        _check_grads(s, grads, ref, ids_np, tol, tag, host)
        _compare("dx", dx.cpu().numpy(), ref["dx"], tol, tag)
        _compare("d_norm_w", host["d_norm_w"], ref["d_norm_w"], tol, tag)
        # the MoE part of dx alone (without the residual) also meets the bar
        _compare("dx - dout", dx.cpu().numpy() - dout.float().cpu().numpy(),
                 ref["dx"] - dout.float().cpu().numpy(), tol, tag)


def _bf16(a):
    return O.bf16_round(np.asarray(a, dtype=np.float64))


def _ulp_bf16(v):
    """one BF16 step at |v|: 2^(e - 7) for |v| in [2^e, 2^(e+1))"""
    a = np.maximum(np.abs(v), 1e-38)
    return np.exp2(np.floor(np.log2(a)) - 7)


def _one_step(name, got, ref, absterms=None):
    """|got - ref| <= one BF16 step of ref plus, for a sum, the FP32 summation
    bound 2^-14 sum|terms| (K u, K <= 1024 terms): an operand both sides round
    to BF16 from values that differ only by FP32 arithmetic"""
    d = np.abs(got.astype(np.float64) - ref)
    bound = _ulp_bf16(ref) * (ref != 0) + 1e-30
    if absterms is not None:
        bound = bound + 2.0 ** -14 * absterms
    bad = d > bound
    assert not bad.any(), f"{name}: {int(bad.sum())} values more than one BF16 step off"


def _fp32_close(name, got, ref):
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = float(np.max(np.abs(got.astype(np.float64) - ref) / (np.abs(ref) + max(rms, 1e-30))))
    assert err <= 1e-4, f"{name}: {err:.3e} off the product of the device's own operands"


@pytest.mark.parametrize("shape,T", [("nano", 5), ("super", 13), ("super", 200)])
def test_backward_products_on_the_device_operands(shape, T):
    from routed_relu_expert_gb300 import _native as N
    s = {"nano": SMALL_NANO, "super": SMALL_SUPER}[shape]
    cfg = M.config_from(s)
    _, (st, dy, dx, grads, bws, x) = layer_backward_parity(s, T)
    ws = st["ws"]
    R, de, I, d, L, S = T * s.top_k, s.d_e, s.d_expert, s.d_model, s.d_latent, s.d_shared

    def fws(region, dt, shape_):
        off, nb = M.workspace_region(cfg, T, region)
        return ws[off:off + nb].view(dt).view(*shape_).float().cpu().numpy().astype(np.float64)

    def fbw(region, shape_):
        off, nb = M.backward_workspace_region(cfg, T, region)
        return bws[off:off + nb].view(torch.bfloat16).view(*shape_).float().cpu().numpy().astype(np.float64)

    w = device_weights(s)
    ow = oracle_weights(w)
    offs = fws(N.MOE_WS_OFFSETS, torch.int32, (-1,)).astype(np.int64)
    rt = fws(N.MOE_WS_ROUTE_TOKEN, torch.int32, (-1,)).astype(np.int64)
    rs = fws(N.MOE_WS_ROUTE_SLOT, torch.int32, (-1,)).astype(np.int64)
    h = fws(N.MOE_WS_H, torch.bfloat16, (R, I))
    x_np = x.float().cpu().numpy().astype(np.float64)
    x_e = fws(N.MOE_WS_X_LATENT, torch.bfloat16, (T, de)) if L else x_np
    dy_np = dy.float().cpu().numpy().astype(np.float64)
    topw = st["topw"].cpu().numpy().astype(np.float64)
    dU = fbw(N.MOE_BWS_DU, (R, de))
    da = fbw(N.MOE_BWS_DA, (R, I))
    dy_r = fbw(N.MOE_BWS_DY_LATENT, (T, L)) if L else dy_np
    if L:
        _one_step("dy_r", dy_r, _bf16(dy_np @ ow["w_lat_up"]), np.abs(dy_np) @ np.abs(ow["w_lat_up"]))
    _one_step("dU", dU, _bf16(topw[rt, rs][:, None] * dy_r[rt]))
    gd = grads["d_down"].cpu().numpy()
    gu = grads["d_up"].cpu().numpy()
    for e in range(s.n_experts):
        a, b = offs[e], offs[e + 1]
        if b == a:
            continue
        down = ow["w_down"][e]
        _one_step(f"da[{e}]", da[a:b], _bf16((dU[a:b] @ down) * 2.0 * np.sqrt(h[a:b])),
                  (np.abs(dU[a:b]) @ np.abs(down)) * 2.0 * np.sqrt(h[a:b]))
        _fp32_close(f"d_down[{e}]", gd[e], dU[a:b].T @ h[a:b])
        _fp32_close(f"d_up[{e}]", gu[e], da[a:b].T @ x_e[rt[a:b]])
    if S:
        das = fbw(N.MOE_BWS_DA_SHARED, (T, S))
        _fp32_close("d_sh_up", grads["d_sh_up"].cpu().numpy(), das.T @ x_np)
    if L:
        dxl = fbw(N.MOE_BWS_DX_LATENT, (T, L))
        _fp32_close("d_lat_down", grads["d_lat_down"].cpu().numpy(), dxl.T @ x_np)

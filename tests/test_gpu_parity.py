"""GPU parity: the CUDA library against the CPU oracle on the same seeded inputs.

Routing (expert ids and per-expert token lists) must match bit for bit, with
the selection checked on the GPU's own FP32 scores; routing weights within
1e-6; logits within 1e-5 of sum_i |x_i W_ei|; the layer output within
2e-2 * RMS for BF16 layers (1e-4 * RMS for FP32 layers)."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from synth import (BF16, NANO_DECODE, NANO_PREFILL, ROUTER_ONLY_GROUPED, SUPER_LATENT, SUPER_NVFP4, TINY_FP32,
                   make_weights, make_x, scaled)

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import routed_relu_expert_gb300 as M
    from gpu_helpers import (check_output, check_route_tables, check_router, device_weights, oracle_weights,
                             run_gpu, to_np, tol_of, ws_table)

SMALL_NANO = scaled(NANO_DECODE, name="nano_scaled", d_model=512, n_experts=32, top_k=4, d_expert=320,
                    d_shared=384, weight_seed=11, tokens=())
SMALL_SUPER = scaled(SUPER_LATENT, name="super_scaled", d_model=512, d_latent=256, n_experts=64, top_k=6,
                     n_group=8, topk_group=4, d_expert=320, d_shared=448, weight_seed=13, tokens=())
SMALL_NVFP4 = scaled(SUPER_LATENT, name="nvfp4_scaled", d_model=512, d_latent=256, n_experts=64, top_k=6,
                     n_group=8, topk_group=4, d_expert=384, d_shared=448, expert_dtype=2, weight_seed=19,
                     tokens=())


def _check_packed_rows(shape, g, x, T):
    """Above 64 BF16 tokens the layer packs its expert input rows for the
    tensor-core kernels: x_packed[j] must be x_e[route_token[j]] bit for bit
    (with NVFP4 experts, the FP16 copy of that BF16 row)."""
    from routed_relu_expert_gb300 import _native as N
    cfg = M.config_from(shape)
    ws = g["ws"]
    de = shape.d_e
    rt = ws_table(ws, cfg, T, N.MOE_WS_ROUTE_TOKEN, torch.int32).long()
    x_e = x if not shape.d_latent else ws_table(ws, cfg, T, N.MOE_WS_X_LATENT, torch.bfloat16).view(T, de)
    want = x_e[rt]
    if shape.expert_dtype == 2:
        want = want.to(torch.float16)
    got = ws_table(ws, cfg, T, N.MOE_WS_X_PACKED, want.dtype).view(-1, de)
    assert torch.equal(got.view(torch.int16), want.contiguous().view(torch.int16))


_E2M1 = np.array([O.e2m1_value(c) for c in range(8)])


def _term_values(codes):
    """Signed E2M1 values of 4-bit codes (a negative zero reads as zero)."""
    return np.where(codes & 8, -1.0, 1.0) * _E2M1[codes & 7]


def _check_fp4_terms(shape, g, x, T, n_terms):
    """On the FP4 tensor path the layer splits the expert input rows and h into
    NVFP4 terms: every code, block scale and row scale must equal the oracle's
    split of the same BF16 rows (both take the decisions in FP32)."""
    from routed_relu_expert_gb300 import _native as N
    cfg = M.config_from(shape)
    ws = g["ws"]
    R, de, I = T * shape.top_k, shape.d_e, shape.d_expert
    nmax = N.ACT_TERMS_MAX
    rt = ws_table(ws, cfg, T, N.MOE_WS_ROUTE_TOKEN, torch.int32).long()
    x_e = x if not shape.d_latent else ws_table(ws, cfg, T, N.MOE_WS_X_LATENT, torch.bfloat16).view(T, de)
    h = ws_table(ws, cfg, T, N.MOE_WS_H, torch.bfloat16).view(R, I)
    for rows, K, rq, rs, rg in ((x_e[rt], de, N.MOE_WS_X_TERMS, N.MOE_WS_X_TERM_SCALES, N.MOE_WS_X_ROW_SCALES),
                                (h, I, N.MOE_WS_H_TERMS, N.MOE_WS_H_TERM_SCALES, N.MOE_WS_H_ROW_SCALES)):
        codes, sf, gg = O.nvfp4_terms(rows.float().cpu().numpy(), n_terms)
        q = ws_table(ws, cfg, T, rq, torch.uint8).view(nmax, R, K // 2)[:n_terms].cpu().numpy()
        got = np.empty((n_terms, R, K), dtype=np.uint8)
        got[..., 0::2], got[..., 1::2] = q & 0xF, q >> 4
        ld = (K // 16 + 15) // 16 * 16
        s_got = ws_table(ws, cfg, T, rs, torch.uint8).view(nmax, R, ld)[:n_terms, :, :K // 16].cpu().numpy()
        g_got = ws_table(ws, cfg, T, rg, torch.float32).cpu().numpy()
        assert np.array_equal(g_got, gg), "row scales differ"
        assert np.array_equal(s_got, sf), f"block scales differ in {np.sum(s_got != sf)} places"
        bad = np.sum(_term_values(got) != _term_values(codes))
        assert bad == 0, f"{bad} term codes differ"


def _parity(shape, T, sample=None, seed_stream=0, chunk=0):
    """Routing of every token (ids bit-exact, weights 1e-6, logits 1e-5), the
    dispatch tables the layer left in its workspace bit-exact, the packed rows
    of the tensor-core path bit-exact, and the output against the oracle on
    every row (or on ``sample`` rows)."""
    w = device_weights(shape)
    x = make_x(shape, T, "cuda", seed_stream)
    g = run_gpu(shape, w, x)
    assert g["err"] == 0
    terms = M.nvfp4_act_terms_for(T)
    fp4_terms = shape.expert_dtype == 2 and terms > 0
    if T > 64 and shape.act_dtype == BF16 and not fp4_terms:
        _check_packed_rows(shape, g, x, T)
    if fp4_terms:
        _check_fp4_terms(shape, g, x, T, terms)
    ws = g.pop("ws")
    g = to_np(g)
    check_route_tables(shape, ws, g["ids"], T)
    del ws
    ow = oracle_weights(w)
    x_np = x.float().cpu().numpy().astype(np.float64)
    # routing on every token
    ids_o, w_o = check_router(shape, x_np, ow, g)
    rows = None
    if sample is not None and sample < T:
        rows = sample if isinstance(sample, np.ndarray) else np.sort(
            np.random.default_rng(T).choice(T, sample, replace=False))
        ids_o, w_o = ids_o[rows], w_o[rows]
    err = check_output(shape, x_np, ow, ids_o, w_o, g["y"], tol_of(shape), rows, chunk=chunk)
    return err, g


@pytest.mark.parametrize("T", [16, 1, 5, 64, 100])
def test_tiny_fp32_layer(T):
    _parity(TINY_FP32, T)


@pytest.mark.parametrize("T", [1, 7, 37, 64, 100, 300])
def test_scaled_nano_layer(T):
    _parity(SMALL_NANO, T)


@pytest.mark.parametrize("T", [1, 13, 64, 200])
def test_scaled_super_latent_layer(T):
    _parity(SMALL_SUPER, T)


@pytest.mark.parametrize("T", [1, 4, 16, 64])
def test_nano_decode_full_size(T):
    _parity(NANO_DECODE, T)


def test_nano_prefill_2048_full():
    _parity(NANO_PREFILL, 2048)


def test_nano_prefill_8192_full():
    """Every token's routing and every output row at T=8192."""
    _parity(NANO_PREFILL, 8192, chunk=4096)


def test_nano_prefill_32768_full():
    """The largest routed workload (196,608 routes, one expert holding most of
    the tokens under the Zipf popularity): routing, dispatch tables and packed
    rows of every token, and every output row."""
    _parity(NANO_PREFILL, 32768, chunk=4096)


@pytest.mark.parametrize("T", [1, 16])
def test_super_latent_full_size(T):
    _parity(SUPER_LATENT, T)


def test_super_latent_256_full():
    _parity(SUPER_LATENT, 256)


def test_super_latent_4096_full():
    _parity(SUPER_LATENT, 4096, chunk=2048)


# 1 and 4 tokens: the FP16 path; 9: the FP4 path; 40 and 64: the FP4 path
# with the dense products on the tensor cores (40: a ragged token tile);
# 65 and 200: the FP16 tensor-core path
@pytest.mark.parametrize("T", [1, 4, 9, 40, 64, 65, 200])
def test_scaled_nvfp4_layer(T):
    _parity(SMALL_NVFP4, T)


@pytest.mark.parametrize("T", [1, 64])
def test_super_nvfp4_full_size(T):
    _parity(SUPER_NVFP4, T)


@pytest.fixture
def act_terms():
    """Sets how NVFP4 experts take their activations for one test."""
    prev = M.set_nvfp4_act_terms(-1)
    yield M.set_nvfp4_act_terms
    M.set_nvfp4_act_terms(prev)


@pytest.mark.parametrize("n", [0, 3, 4])
@pytest.mark.parametrize("T", [1, 9, 200])
def test_scaled_nvfp4_layer_every_activation_form(act_terms, n, T):
    """The FP16 path (0) and three or four terms on the FP4 tensor path, at
    one token, decode and prefill sizes, against the exact oracle."""
    act_terms(n)
    _parity(SMALL_NVFP4, T, seed_stream=n)


@pytest.mark.parametrize("n", [0, 3])
def test_super_nvfp4_on_the_paths_the_default_skips(act_terms, n):
    """Full-size Super NVFP4 layers on the path the default does not take at
    that size, every row against the oracle: the FP16 path at 64 tokens and
    the FP4 path at 8192 (the default's paths are covered by the full-size
    tests above)."""
    act_terms(n)
    if n == 0:
        _parity(SUPER_NVFP4, 64, chunk=64)        # the FP16 path at the decode size the default gives the FP4 path
    else:
        _parity(SUPER_NVFP4, 8192, chunk=8192)    # the FP4 path at the prefill size the default gives the FP16 path


@pytest.mark.parametrize("n", [1, 2])
@pytest.mark.parametrize("T", [9, 200])
def test_few_term_layer_against_the_oracle_with_the_same_terms(act_terms, n, T):
    """One term (plain W4A4) and two terms miss the exact layer by more than
    the NVFP4 tolerance; each equals the oracle evaluated with its expert
    inputs and h replaced by their n-term NVFP4 forms."""
    act_terms(n)
    shape = SMALL_NVFP4
    w = device_weights(shape)
    x = make_x(shape, T, "cuda", 7)
    g = run_gpu(shape, w, x)
    assert g["err"] == 0
    _check_fp4_terms(shape, g, x, T, n)
    g.pop("ws")
    g = to_np(g)
    ow = oracle_weights(w)
    x_np = x.float().cpu().numpy().astype(np.float64)
    ids_o, w_o = check_router(shape, x_np, ow, g)
    ref = O.layer_forward(x_np, ow, ids_o, w_o, shape.n_experts, bf16_points=True, act_terms=n)["y"]
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = float(np.max(np.abs(g["y"].astype(np.float64) - ref))) / rms
    assert err <= 5e-2, f"max |y - y_ref| = {err:.3e} RMS"


def test_super_nvfp4_8192_full():
    _parity(SUPER_NVFP4, 8192, chunk=8192)


def test_router_grouped_case_from_the_router_parity_test():
    """128 experts, top-6, eight groups keeping three: the router parity case
    of page "Nemotron Is Not One Circuit", section "What CKE Has Actually
    Established"; exact ids and weights within 1e-6."""
    shape = ROUTER_ONLY_GROUPED
    w = device_weights(shape)
    for T in (1, 64, 333):
        x = make_x(shape, T, "cuda")
        cfg = M.config_from(shape)
        ws = M.new_workspace(cfg, T)
        ids = torch.empty((T, shape.top_k), dtype=torch.int32, device="cuda")
        topw = torch.empty((T, shape.top_k), dtype=torch.float32, device="cuda")
        logits = torch.empty((T, shape.n_experts), dtype=torch.float32, device="cuda")
        scores = torch.empty_like(logits)
        M.moe_router(cfg, x, w["w_router"], w["bias"], ids, topw, ws, logits, scores)
        torch.cuda.synchronize()
        g = to_np({"ids": ids, "topw": topw, "logits": logits, "scores": scores})
        ow = oracle_weights({"w_router": w["w_router"], "bias": w["bias"]})
        check_router(shape, x.float().cpu().numpy().astype(np.float64), ow, g)


@pytest.mark.parametrize("T,E,K", [(1, 8, 2), (64, 128, 6), (37, 512, 22), (2048, 128, 6), (700, 64, 6)])
def test_dispatch_is_bit_exact(T, E, K):
    from synth import MoEShape
    shape = MoEShape("dispatch", 256, 0, E, K, 1, 1, 128, 0, 1.0, tokens=())
    cfg = M.config_from(shape)
    rng = np.random.default_rng(T + E)
    p = rng.zipf(1.5, E).astype(np.float64)
    p /= p.sum()
    ids_np = np.stack([rng.choice(E, K, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    ids = torch.from_numpy(ids_np).cuda()
    x = torch.randn((T, 256), device="cuda").to(torch.bfloat16)
    ws = M.new_workspace(cfg, T)
    R = T * K
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    rt = torch.empty(R, dtype=torch.int32, device="cuda")
    rs = torch.empty(R, dtype=torch.int32, device="cuda")
    tsr = torch.empty((T, K), dtype=torch.int32, device="cuda")
    xp = torch.empty((R, 256), dtype=torch.bfloat16, device="cuda")
    M.moe_clear_device_error(ws)          # a fresh workspace holds garbage; step calls do not clear it
    M.moe_dispatch(cfg, ids, counts, offsets, rt, rs, tsr, ws, x_e=x, x_packed=xp)
    torch.cuda.synchronize()
    ref = O.dispatch(ids_np, E)
    assert np.array_equal(counts.cpu().numpy(), ref["counts"])
    assert np.array_equal(offsets.cpu().numpy(), ref["offsets"])
    assert np.array_equal(rt.cpu().numpy(), ref["route_token"])
    assert np.array_equal(rs.cpu().numpy(), ref["route_slot"])
    assert np.array_equal(tsr.cpu().numpy(), ref["token_slot_row"])
    assert torch.equal(xp, x[torch.from_numpy(ref["route_token"]).cuda()])
    assert M.moe_get_device_error(ws) == 0


@pytest.mark.parametrize("case", ["decode", "prefill"])
def test_step_entry_points_reproduce_layer_forward_bit_for_bit(case):
    # (the NVFP4 layer runs its decode GEMVs on FP16 copies of the activations,
    # the step entry points on the BF16 tensors: the same values either way.
    # At prefill sizes moe_experts_up is given x_e only and gathers the rows
    # itself for the tensor-core kernel.)
    cases = (((SMALL_NANO, 37), (SMALL_SUPER, 13), (SMALL_NVFP4, 9)) if case == "decode"
             else ((SMALL_NANO, 300), (SMALL_SUPER, 200)))
    for shape, T in cases:
        w = device_weights(shape)
        x = make_x(shape, T, "cuda", 3)
        cfg = M.config_from(shape)
        layer = M.MoELayer(cfg, w)
        y_ref = layer.forward(x).clone()
        E, K, de = shape.n_experts, shape.top_k, shape.d_e
        ws = M.new_workspace(cfg, T)
        ids = torch.empty((T, K), dtype=torch.int32, device="cuda")
        topw = torch.empty((T, K), dtype=torch.float32, device="cuda")
        M.moe_router(cfg, x, w["w_router"], w["bias"], ids, topw, ws)
        x_e = x
        if shape.d_latent:
            x_e = torch.empty((T, de), dtype=x.dtype, device="cuda")
            M.moe_latent_down(cfg, x, layer.weights, x_e, ws)
        counts = torch.empty(E, dtype=torch.int32, device="cuda")
        offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
        rt = torch.empty(T * K, dtype=torch.int32, device="cuda")
        rs = torch.empty(T * K, dtype=torch.int32, device="cuda")
        tsr = torch.empty((T, K), dtype=torch.int32, device="cuda")
        M.moe_dispatch(cfg, ids, counts, offsets, rt, rs, tsr, ws)
        h = torch.empty((T * K, shape.d_expert), dtype=x.dtype, device="cuda")
        M.moe_experts_up(cfg, T, rt, offsets, layer.weights, h, ws, x_e=x_e)
        y_r = torch.empty((T, de), dtype=torch.float32, device="cuda")
        M.moe_experts_down_combine(cfg, T, h, offsets, rt, rs, tsr, topw, layer.weights, y_r, ws)
        y = torch.empty_like(x)
        M.moe_shared(cfg, x, layer.weights, y, ws, y_routed=y_r)
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref)


def test_runs_are_bit_identical():
    shape = NANO_DECODE
    w = device_weights(shape)
    x = make_x(shape, 64, "cuda", 5)
    layer = M.MoELayer(M.config_from(shape), w)
    ys = [layer.forward(x).clone() for _ in range(3)]
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[1], ys[2])


def test_zero_tokens_is_a_no_op():
    shape = SMALL_NANO
    layer = M.MoELayer(M.config_from(shape), device_weights(shape))
    x = torch.empty((0, shape.d_model), dtype=torch.bfloat16, device="cuda")
    y = layer.forward(x)
    assert y.shape == (0, shape.d_model)


def test_nan_input_sets_the_nonfinite_bit_and_keeps_ids_in_range():
    shape = SMALL_NANO
    w = device_weights(shape)
    x = make_x(shape, 8, "cuda")
    x[3, 5] = float("nan")
    g = run_gpu(shape, w, x)
    assert g["err"] & M.MOE_DEVERR_NONFINITE
    ids = g["ids"].cpu().numpy()
    assert ids.min() >= 0 and ids.max() < shape.n_experts
    assert all(len(set(r)) == shape.top_k for r in ids.tolist())


def test_out_of_range_ids_are_flagged_and_skipped():
    from synth import MoEShape
    E, K, T = 16, 2, 10
    shape = MoEShape("bad_ids", 256, 0, E, K, 1, 1, 128, 0, 1.0, tokens=())
    cfg = M.config_from(shape)
    ids_np = np.tile(np.array([[0, 1]], dtype=np.int32), (T, 1))
    ids_np[4, 1] = E            # out of range
    ids_np[6, 0] = -3
    ids = torch.from_numpy(ids_np).cuda()
    ws = M.new_workspace(cfg, T)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    rt = torch.full((T * K,), -7, dtype=torch.int32, device="cuda")
    rs = torch.empty(T * K, dtype=torch.int32, device="cuda")
    tsr = torch.empty((T, K), dtype=torch.int32, device="cuda")
    M.moe_clear_device_error(ws)
    M.moe_dispatch(cfg, ids, counts, offsets, rt, rs, tsr, ws)
    assert M.moe_get_device_error(ws) & M.MOE_DEVERR_EXPERT_ID
    assert int(counts.sum()) == T * K - 2
    t = tsr.cpu().numpy()
    assert t[4, 1] == -1 and t[6, 0] == -1


@pytest.mark.parametrize("T", [1, 9, 200])
def test_nvfp4_rows_beyond_fp16_range(T):
    """Expert input rows scaled by 2^16 (exact in BF16, beyond FP16's 65504):
    the FP16 path (under 8 tokens; above 64 tokens) flags MOE_DEVERR_RANGE instead
    of returning silent infinities; the FP4 path (8..64 tokens) carries the
    magnitude in each row's FP32 scale and still matches the oracle."""
    from routed_relu_expert_gb300 import _native as N
    shape = SMALL_NVFP4
    w = device_weights(shape)
    x = (make_x(shape, T, "cuda").float() * 65536.0).to(torch.bfloat16)
    g = run_gpu(shape, w, x)
    ws = g.pop("ws")
    if M.nvfp4_act_terms_for(T) == 0:
        assert g["err"] & N.MOE_DEVERR_RANGE, f"FP16 path at T={T} did not flag the range"
        return
    assert g["err"] == 0
    g = to_np(g)
    assert np.all(np.isfinite(g["y"]))
    ow = oracle_weights(w)
    x_np = x.float().cpu().numpy().astype(np.float64)
    ids_o, w_o = check_router(shape, x_np, ow, g)
    check_output(shape, x_np, ow, ids_o, w_o, g["y"], tol_of(shape))


@pytest.mark.parametrize("T,groups", [(1, 1), (1, 8), (3, 1), (3, 8), (40, 1), (40, 8), (100, 8)])
def test_topk_above_eight_with_exact_ties(T, groups):
    """K = 12 of E = 256 (the selection-by-threshold path for K > 8): router
    rows duplicated in pairs and a zero bias give exactly equal scores, so
    every choice crosses ties; ids must match the oracle's selection (lower id
    first) on the GPU's own scores, through the fused tiny kernel (T = 1: the
    whole CTA selects the token of this 256-expert router; T = 3: a warp a
    token) and the per-token selection kernel."""
    from synth import make_weights as mw
    shape = scaled(NANO_DECODE, name=f"ties_{groups}", d_model=256, n_experts=256, top_k=12, n_group=groups,
                   topk_group=4 if groups > 1 else 1, d_expert=128, d_shared=0, weight_seed=67, tokens=())
    w = mw(shape, "cuda")
    w["w_router"] = w["w_router"][0::2].repeat_interleave(2, dim=0).contiguous()
    w["bias"] = torch.zeros_like(w["bias"])
    x = make_x(shape, T, "cuda")
    g = run_gpu(shape, w, x)
    assert g["err"] == 0
    g.pop("ws")
    g = to_np(g)
    ow = oracle_weights(w)
    s = g["scores"]
    assert np.array_equal(s[:, 0::2], s[:, 1::2])          # every score tied with its pair
    check_router(shape, x.float().cpu().numpy().astype(np.float64), ow, g)


@pytest.mark.parametrize("T,d_model", [(4, 1024), (5, 1024), (8, 1024), (9, 1024), (16, 1024), (17, 1024),
                                       (32, 1024), (33, 1024), (64, 1024), (6, 1088), (40, 1088)])
def test_wide_router_logits_every_tile_height(T, d_model):
    """Routers with E >= 256 at 4..64 tokens: at 5-8 tokens the logits come
    from rows staged per 8 experts x 8 tokens, above 32 tokens per 16 x 16,
    otherwise from the per-2-experts kernel; logits within 1e-5 of sum |x W|,
    ids and weights against the oracle on the GPU scores, on both sides of
    every switch.  A hidden width of 1088 leaves a last K chunk of 64 values."""
    shape = scaled(SUPER_LATENT, name="wide_router", d_model=d_model, d_latent=256, n_experts=256, top_k=12,
                   n_group=8, topk_group=4, d_expert=128, d_shared=0, weight_seed=71, tokens=())
    w = device_weights(shape)
    x = make_x(shape, T, "cuda")
    g = run_gpu(shape, w, x)
    assert g["err"] == 0
    g.pop("ws")
    g = to_np(g)
    check_router(shape, x.float().cpu().numpy().astype(np.float64), oracle_weights(w), g)


@pytest.mark.parametrize("T", [7, 20, 40])
def test_wide_router_fp32_layer(T):
    """An FP32 layer with a 256-expert router: at 7 and 40 tokens the router
    reads FP32 token rows through the staged kernels, at 20 through the
    per-2-experts kernel; routing and the whole layer against the oracle."""
    from synth import TINY_FP32
    shape = scaled(TINY_FP32, name="wide_router_fp32", d_model=512, n_experts=256, top_k=8, n_group=8,
                   topk_group=4, d_expert=128, d_shared=256, weight_seed=73, tokens=())
    _parity(shape, T)

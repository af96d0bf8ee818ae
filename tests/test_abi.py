"""The C ABI library: it loads, exports every entry point the header declares,
and rejects bad arguments on the host before enqueuing anything (no GPU
needed: every call here returns before its first CUDA call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_gb300.h")


@pytest.fixture(scope="module")
def lib():
    from routed_relu_expert_gb300 import build
    build.build()
    from routed_relu_expert_gb300 import _native
    return _native.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_entry_point(lib):
    names = _declared_functions()
    assert "moe_layer_forward" in names and len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    from routed_relu_expert_gb300 import EXPORTS
    assert sorted(EXPORTS) == names


def test_struct_layout_matches_header(lib):
    from routed_relu_expert_gb300 import MoeConfig, MoeWeights
    assert ctypes.sizeof(MoeConfig) == 12 * 4
    # one pointer per member the header declares in moe_weights_t, in order
    text = open(HEADER).read()
    body = text[text.index("typedef struct moe_weights {"):text.index("} moe_weights_t;")]
    members = re.findall(r"\*\s*(w_[a-z_]+|router_bias)\s*;", body)
    assert [f[0] for f in MoeWeights._fields_] == members
    assert ctypes.sizeof(MoeWeights) == len(members) * 8
    from routed_relu_expert_gb300._native import MoeGrads
    body = text[text.index("typedef struct moe_grads {"):text.index("} moe_grads_t;")]
    members = re.findall(r"\*\s*(d_[a-z_]+)\s*;", body)
    assert [f[0] for f in MoeGrads._fields_] == members


def _cfg(**kw):
    from routed_relu_expert_gb300 import make_config
    base = dict(d_model=256, n_experts=8, top_k=2, d_expert=128, d_shared=256, routed_scaling_factor=2.5)
    base.update(kw)
    return make_config(**base)


def test_config_validation(lib):
    from routed_relu_expert_gb300 import _native as N
    ok = _cfg()
    assert lib.moe_check_config(ctypes.byref(ok)) == N.MOE_OK
    bad = [
        _cfg(top_k=9),                               # K > E
        _cfg(n_experts=0),
        _cfg(n_group=3),                             # E % G != 0
        _cfg(n_group=4, topk_group=5),               # TG > G
        _cfg(n_group=8, topk_group=1, top_k=2),      # groups of one expert
        _cfg(n_group=4, topk_group=1, top_k=3),      # K > TG * E/G
        _cfg(top_k=33, n_experts=64),
        _cfg(norm_topk_prob=2),
        _cfg(routed_scaling_factor=float("nan")),
        _cfg(act_dtype=7),
    ]
    for c in bad:
        assert lib.moe_check_config(ctypes.byref(c)) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_check_config(ctypes.byref(_cfg(d_model=250))) == N.MOE_ERR_UNSUPPORTED
    # F32 experts need F32 activations
    assert lib.moe_check_config(ctypes.byref(_cfg(expert_dtype=N.MOE_DT_F32))) == N.MOE_ERR_UNSUPPORTED


def test_workspace_size_grows_with_tokens_and_rejects_short_buffers(lib):
    from routed_relu_expert_gb300 import _native as N
    c = _cfg()
    sizes = [lib.moe_workspace_bytes(ctypes.byref(c), T) for T in (0, 1, 16, 1000)]
    assert sizes[0] > 0 and sizes == sorted(sizes) and sizes[3] > sizes[2]
    assert all(s % 256 == 0 for s in sizes)
    assert lib.moe_workspace_bytes(ctypes.byref(_cfg(top_k=9)), 4) == 0
    # a workspace one byte short is refused before any device work
    fake = ctypes.c_void_p(1 << 20)            # never dereferenced: the size check comes first
    w = N.MoeWeights()
    st = lib.moe_layer_forward(ctypes.byref(c), 16, fake, ctypes.byref(w), fake, None, None, None, None,
                               fake, ctypes.c_size_t(sizes[2] - 1), None)
    assert st == N.MOE_ERR_WORKSPACE


def test_null_and_misaligned_pointers_are_refused(lib):
    from routed_relu_expert_gb300 import _native as N
    c = _cfg()
    n = lib.moe_workspace_bytes(ctypes.byref(c), 4)
    ws = ctypes.c_void_p(1 << 20)
    good = ctypes.c_void_p(1 << 21)
    mis = ctypes.c_void_p((1 << 21) + 4)
    w = N.MoeWeights()
    args = lambda x, y: (ctypes.byref(c), 4, x, ctypes.byref(w), y, None, None, None, None, ws, n, None)
    assert lib.moe_layer_forward(*args(None, good)) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_forward(*args(mis, good)) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_forward(*args(good, good)) == N.MOE_ERR_INVALID_ARG   # weights missing
    assert lib.moe_router(ctypes.byref(c), 4, good, None, None, None, None, good, good, ws, n, None) == \
        N.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch(ctypes.byref(c), 4, good, None, good, good, good, good, None, None, ws, n, None) == \
        N.MOE_ERR_INVALID_ARG
    assert lib.moe_latent_down(ctypes.byref(c), 4, good, ctypes.byref(w), good, ws, n, None) == \
        N.MOE_ERR_INVALID_ARG                                                 # not a latent layer
    # zero tokens: nothing to do, nothing touched
    assert lib.moe_layer_forward(ctypes.byref(c), 0, None, ctypes.byref(w), None, None, None, None, None,
                                 None, 0, None) == N.MOE_OK
    assert lib.moe_get_device_error(None, None, None) == N.MOE_ERR_INVALID_ARG


def test_status_strings(lib):
    for s in range(6):
        assert lib.moe_status_string(s)
    assert lib.moe_version() >= 100


def test_noalloc_limits_match_header():
    """The binding's copies of the static-scratch limits equal the header's."""
    from routed_relu_expert_gb300 import _native as N
    text = open(HEADER).read()
    for name in ("MOE_NOALLOC_MAX_ROUTER_ELEMS", "MOE_NOALLOC_MAX_SPLIT_ELEMS"):
        m = re.search(r"#define\s+" + name + r"\s+(\d+)", text)
        assert m, name
        assert int(m.group(1)) == getattr(N, name)


def test_workspace_regions_lie_inside_the_workspace(lib):
    """Every route table moe_workspace_region names fits in moe_workspace_bytes,
    with the sizes the header states, and no two overlap."""
    from routed_relu_expert_gb300 import _native as N
    import routed_relu_expert_gb300 as M
    from synth import NANO_DECODE, SUPER_NVFP4
    for shape, T in ((NANO_DECODE, 1), (NANO_DECODE, 300), (SUPER_NVFP4, 65)):
        cfg = M.config_from(shape)
        total = M.workspace_bytes(cfg, T)
        E, K, R = shape.n_experts, shape.top_k, T * shape.top_k
        sizes = {N.MOE_WS_COUNTS: E * 4, N.MOE_WS_OFFSETS: (E + 1) * 4, N.MOE_WS_ROUTE_TOKEN: R * 4,
                 N.MOE_WS_ROUTE_SLOT: R * 4, N.MOE_WS_TOKEN_SLOT_ROW: R * 4, N.MOE_WS_TOPK_IDS: R * 4,
                 N.MOE_WS_TOPK_W: R * 4, N.MOE_WS_LOGITS: T * E * 4, N.MOE_WS_SCORES: T * E * 4,
                 N.MOE_WS_X_LATENT: T * shape.d_latent * 2, N.MOE_WS_X_PACKED: R * shape.d_e * 2}
        spans = []
        for region, nbytes in sizes.items():
            off, n = M.workspace_region(cfg, T, region)
            assert n == nbytes and off % 256 == 0 and off + n <= total
            if n:
                spans.append((off, off + n))
        spans.sort()
        assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))
        off = ctypes.c_size_t(0)
        assert lib.moe_workspace_region(ctypes.byref(cfg), T, 99, ctypes.byref(off), ctypes.byref(off)) == \
            N.MOE_ERR_INVALID_ARG


def test_block_sparse_and_backward_arguments_are_checked_before_any_work(lib):
    """The block, sparse-down and backward entry points refuse bad arguments
    and unsupported configurations on the host, before any CUDA call (these
    addresses are never dereferenced)."""
    from routed_relu_expert_gb300 import _native as N
    c = _cfg()
    n = lib.moe_workspace_bytes(ctypes.byref(c), 4)
    nb = lib.moe_backward_workspace_bytes(ctypes.byref(c), 4)
    assert n > 0 and nb > 0
    ws, good = ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 21)
    P = [ctypes.c_void_p((1 << 22) + 256 * i) for i in range(16)]
    w = N.MoeWeights(w_router=P[0], w_up=P[1], w_down=P[2], w_sh_up=P[3], w_sh_down=P[4])
    # block: a negative or non-finite epsilon, a missing norm weight, an output overlapping x
    blk = lambda x, g, eps, out, xn=None: lib.moe_block_forward(ctypes.byref(c), 4, x, g, ctypes.c_float(eps),
                                                               ctypes.byref(w), out, xn, None, None, None, None,
                                                               ws, n, None)
    assert blk(good, P[5], -1.0, P[6]) == N.MOE_ERR_INVALID_ARG
    assert blk(good, P[5], float("nan"), P[6]) == N.MOE_ERR_INVALID_ARG
    assert blk(good, None, 1e-5, P[6]) == N.MOE_ERR_INVALID_ARG
    assert blk(good, P[5], 1e-5, ctypes.c_void_p((1 << 21) + 256)) == N.MOE_ERR_INVALID_ARG   # partial overlap
    assert blk(good, P[5], 1e-5, P[6], good) == N.MOE_ERR_INVALID_ARG                          # xn is x
    # sparse down: FP32 layers and unfit shapes are refused
    v, s = ctypes.c_size_t(0), ctypes.c_size_t(0)
    f32 = _cfg(act_dtype=N.MOE_DT_F32, expert_dtype=N.MOE_DT_F32)
    assert lib.moe_sparse_down_bytes(ctypes.byref(f32), ctypes.byref(v), ctypes.byref(s)) == N.MOE_ERR_UNSUPPORTED
    assert lib.moe_sparse_down_bytes(ctypes.byref(c), ctypes.byref(v), ctypes.byref(s)) == N.MOE_OK
    assert v.value == 8 * 256 * 128 * 2 and s.value == 0
    fp4 = _cfg(expert_dtype=N.MOE_DT_NVFP4)
    assert lib.moe_sparse_down_bytes(ctypes.byref(fp4), ctypes.byref(v), ctypes.byref(s)) == N.MOE_OK
    assert v.value == 8 * 256 * 128 // 2 and s.value == 8 * 256 * 128 // 16
    # backward: BF16 layers only, a big enough scratch, every saved tensor given
    g = N.MoeGrads()
    bwd = lambda cfg, ids, nbw: lib.moe_layer_backward(ctypes.byref(cfg), 4, good, ctypes.byref(w), P[7], ids, P[8],
                                                       P[9], P[10], ctypes.byref(g), ws,
                                                       lib.moe_workspace_bytes(ctypes.byref(cfg), 4), P[11], nbw,
                                                       None)
    assert bwd(fp4, P[12], 1 << 30) == N.MOE_ERR_UNSUPPORTED
    assert bwd(c, P[12], nb - 1) == N.MOE_ERR_WORKSPACE
    assert bwd(c, None, nb) == N.MOE_ERR_INVALID_ARG
    # regions of the backward scratch lie inside it
    for region in range(6):
        off, nbytes = ctypes.c_size_t(0), ctypes.c_size_t(0)
        assert lib.moe_backward_workspace_region(ctypes.byref(c), 4, region, ctypes.byref(off),
                                                 ctypes.byref(nbytes)) == N.MOE_OK
        assert off.value % 256 == 0 and off.value + nbytes.value <= nb
    assert lib.moe_backward_workspace_region(ctypes.byref(c), 4, 6, ctypes.byref(off), ctypes.byref(nbytes)) == \
        N.MOE_ERR_INVALID_ARG

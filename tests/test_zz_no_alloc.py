"""The router entry point that allocates nothing (moe_router_noalloc).

Some callers cannot allocate device memory when they call the layer: their
host framework's pool already owns the device, their serving loop forbids
allocation once started, or they enqueue work where cudaMalloc is not
permitted.  This entry point keeps its scratch in a static device array of the
library instead of a workspace.  The test calls it through the C ABI and
checks it against moe_router (the workspace entry point) on two calls in a
row (it runs the same kernels, so ids must be equal and weights within the
1e-6 the other router tests use), checks its choice against the oracle's
selection on the same FP32 scores, checks that a call leaves the device's free
memory and torch's allocator untouched, and checks that an oversized call is
refused before any work.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from synth import NANO_DECODE, ROUTER_ONLY_GROUPED, SUPER_LATENT, make_x, router_params

pytestmark = pytest.mark.gpu

TOL_W = 1e-6


def _lib():
    import routed_relu_expert_gb300 as M
    return M, M.load()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(M, lib, cfg, x, wr, b, ids, topw):
    return lib.moe_router_noalloc(ctypes.byref(cfg), x.shape[0], _ptr(x), _ptr(wr), _ptr(b), _ptr(ids),
                                  _ptr(topw), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


# (SUPER_LATENT, 256): T * n_experts is exactly the scratch's limit, with the
# 512-expert split router matrix and the K-split slabs in use
@pytest.mark.parametrize("shape,T", [(NANO_DECODE, 64), (SUPER_LATENT, 16), (ROUTER_ONLY_GROUPED, 1),
                                     (NANO_DECODE, 1024), (SUPER_LATENT, 256)])
def test_noalloc_router_matches_workspace_router_on_two_calls(shape, T):
    M, lib = _lib()
    cfg = M.config_from(shape)
    rp = router_params(shape)
    wr, b = rp["w_router"].cuda(), rp["bias"].cuda()
    K, E = shape.top_k, shape.n_experts
    for call in range(2):                      # two calls in a row, different inputs
        x = make_x(shape, T, "cuda", stream_id=call)
        ids_ref = torch.empty((T, K), dtype=torch.int32, device="cuda")
        w_ref = torch.empty((T, K), dtype=torch.float32, device="cuda")
        scores = torch.empty((T, E), dtype=torch.float32, device="cuda")
        ws = M.new_workspace(cfg, T)
        M.moe_router(cfg, x, wr, b, ids_ref, w_ref, ws, scores=scores)
        ids = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
        topw = torch.full((T, K), -1.0, dtype=torch.float32, device="cuda")
        assert _noalloc(M, lib, cfg, x, wr, b, ids, topw) == 0
        torch.cuda.synchronize()
        assert torch.equal(ids, ids_ref)
        assert float((topw - w_ref).abs().max()) <= TOL_W
        # the oracle's selection on the same FP32 scores (the workspace router's export)
        ids_o, w_o = O.route(scores.cpu().numpy(), rp["bias"].numpy(), shape.n_group, shape.topk_group, K,
                             shape.norm_topk_prob, shape.routed_scaling_factor)
        assert np.array_equal(ids.cpu().numpy(), ids_o)
        assert np.max(np.abs(topw.cpu().numpy().astype(np.float64) - w_o)) <= TOL_W


def test_noalloc_router_call_allocates_nothing():
    """After a first (set-up) call, a call changes neither the device's free
    memory nor torch's allocator."""
    M, lib = _lib()
    shape, T = NANO_DECODE, 1024               # the tensor-core path with the split matrix and K parts
    cfg = M.config_from(shape)
    rp = router_params(shape)
    wr, b = rp["w_router"].cuda(), rp["bias"].cuda()
    x = make_x(shape, T, "cuda")
    ids = torch.empty((T, shape.top_k), dtype=torch.int32, device="cuda")
    topw = torch.empty((T, shape.top_k), dtype=torch.float32, device="cuda")
    assert _noalloc(M, lib, cfg, x, wr, b, ids, topw) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(3):
        assert _noalloc(M, lib, cfg, x, wr, b, ids, topw) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_allocated() == alloc0


def test_noalloc_router_refuses_sizes_beyond_its_scratch():
    M, lib = _lib()
    from routed_relu_expert_gb300 import _native as N
    shape = SUPER_LATENT                       # 512 experts
    cfg = M.config_from(shape)
    T = N.MOE_NOALLOC_MAX_ROUTER_ELEMS // shape.n_experts + 1
    rp = router_params(shape)
    wr, b = rp["w_router"].cuda(), rp["bias"].cuda()
    x = torch.zeros((T, shape.d_model), dtype=torch.bfloat16, device="cuda")
    ids = torch.full((T, shape.top_k), -1, dtype=torch.int32, device="cuda")
    topw = torch.zeros((T, shape.top_k), dtype=torch.float32, device="cuda")
    assert _noalloc(M, lib, cfg, x, wr, b, ids, topw) == N.MOE_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int(ids.max()) == -1                # nothing was written

"""The router entry point that allocates nothing (moe_router_noalloc).

Some callers cannot allocate device memory when they call the layer: their
host framework's pool already owns the device, their serving loop forbids
allocation once started, or they enqueue work where cudaMalloc is not
permitted.  This entry point keeps its scratch in a static device array of the
library instead of a workspace.  The test calls it through the C ABI and
checks it against moe_router (the workspace entry point) on two calls in a
row (it runs the same kernels, so ids must be equal and weights within the
1e-6 the other router tests use), and checks that an oversized call is
refused before any work.
"""
import ctypes

import numpy as np
import pytest
import torch

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


@pytest.mark.parametrize("shape,T", [(NANO_DECODE, 64), (SUPER_LATENT, 16), (ROUTER_ONLY_GROUPED, 1),
                                     (NANO_DECODE, 1024)])
def test_noalloc_router_matches_workspace_router_on_two_calls(shape, T):
    M, lib = _lib()
    cfg = M.config_from(shape)
    rp = router_params(shape)
    wr, b = rp["w_router"].cuda(), rp["bias"].cuda()
    K = shape.top_k
    for call in range(2):                      # two calls in a row, different inputs
        x = make_x(shape, T, "cuda", stream_id=call)
        ids_ref = torch.empty((T, K), dtype=torch.int32, device="cuda")
        w_ref = torch.empty((T, K), dtype=torch.float32, device="cuda")
        ws = M.new_workspace(cfg, T)
        M.moe_router(cfg, x, wr, b, ids_ref, w_ref, ws)
        ids = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
        topw = torch.full((T, K), -1.0, dtype=torch.float32, device="cuda")
        assert _noalloc(M, lib, cfg, x, wr, b, ids, topw) == 0
        torch.cuda.synchronize()
        assert torch.equal(ids, ids_ref)
        assert float((topw - w_ref).abs().max()) <= TOL_W


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

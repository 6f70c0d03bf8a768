"""moe_forward_static: the forward for callers that cannot allocate device memory.

Such callers (a plugin whose host inference engine owns every device allocation, or a
loop that must not call cudaMalloc because it can synchronise the device) get the
scratch from a fixed array inside the library. This file is collected last on purpose,
so a failure here comes after every other test has run; it also passes on its own in a
fresh process. The calls go through the C ABI directly.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

Y_TOL = 2e-2   # the bf16 output tolerance used by the other parity tests


def _inputs(T, H, I, E, k, shared_I, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16).cuda()
    w13 = (torch.randn(E, 2 * I, H, generator=g) * H ** -0.5).to(torch.bfloat16).cuda()
    w2 = (torch.randn(E, H, I, generator=g) * I ** -0.5).to(torch.bfloat16).cuda()
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).int().cuda()
    sc = torch.rand(T, k, generator=g).float().cuda()
    w13s = w2s = None
    if shared_I:
        w13s = (torch.randn(2 * shared_I, H, generator=g) * H ** -0.5).to(torch.bfloat16).cuda()
        w2s = (torch.randn(H, shared_I, generator=g) * shared_I ** -0.5).to(torch.bfloat16).cuda()
    return x, ids, sc, w13, w2, w13s, w2s


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("T,H,I,E,k,shared_I", [(64, 2048, 768, 128, 8, 0),
                                                 (300, 512, 256, 16, 4, 256)])
def test_static_scratch_forward_matches_workspace_forward(T, H, I, E, k, shared_I):
    import mixture_experts_layer_03_gb300 as moe
    lib = moe._lib
    x, ids, sc, w13, w2, w13s, w2s = _inputs(T, H, I, E, k, shared_I, seed=T + E)
    p = moe.make_problem(T, H, I, E, k, shared_I)
    assert moe.moe_workspace_bytes(p) <= moe.MOE_STATIC_SCRATCH_BYTES
    ws = moe.alloc_workspace(p)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    y_ref = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    st = lib.moe_forward(ctypes.byref(p), _p(x), _p(ids), _p(sc), _p(w13), _p(w2), _p(w13s),
                         _p(w2s), _p(y_ref), ws.ptr, ws.nbytes, stream)
    assert st == moe.MOE_OK, lib.moe_last_error()
    ref = y_ref.float().cpu().numpy()
    for _ in range(2):   # two calls in a row: the scratch keeps the previous call's contents
        y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = lib.moe_forward_static(ctypes.byref(p), _p(x), _p(ids), _p(sc), _p(w13), _p(w2),
                                    _p(w13s), _p(w2s), _p(y), stream)
        assert st == moe.MOE_OK, lib.moe_last_error()
        torch.cuda.synchronize()
        got = y.float().cpu().numpy()
        assert np.isfinite(got).all()
        err = np.abs(got - ref).max()
        assert err <= Y_TOL * np.abs(ref).max(), err


def test_static_scratch_rejects_problems_that_do_not_fit():
    import mixture_experts_layer_03_gb300 as moe
    p = moe.make_problem(T=4096, H=4096, I=14336, E=8, k=2)
    assert moe.moe_workspace_bytes(p) > moe.MOE_STATIC_SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: the size check comes first
    st = moe._lib.moe_forward_static(ctypes.byref(p), fake, fake, fake, fake, fake, None, None,
                                     fake, None)
    assert st == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    assert b"static scratch" in moe._lib.moe_last_error()

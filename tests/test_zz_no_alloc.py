"""moe_forward_static: the forward for callers that cannot allocate device memory.

Such callers (a plugin whose host inference engine owns every device allocation, or a
loop that must not call cudaMalloc because it can synchronise the device) get the
scratch from a fixed array inside the library. This file is collected last on purpose,
so a failure here comes after every other test has run; it also passes on its own in a
fresh process. The calls go through the C ABI directly.

Each shape is checked against the CPU oracle (fp64) at the bf16 output tolerance of the
other parity tests, and byte for byte against moe_forward with a caller workspace (the
same kernels, so the scratch's base and layout must not change a single bit), on two
calls in a row.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle

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


def _np64(t):
    return None if t is None else t.cpu().double().numpy()


@pytest.mark.parametrize("T,H,I,E,k,shared_I", [
    (64, 2048, 768, 128, 8, 0),     # a decode batch: narrow single-SM tiles
    (300, 512, 256, 16, 4, 256),    # shared expert, row-by-row copy of the permute step
    (2048, 256, 128, 8, 2, 0),      # 2048 tokens: the token-major row copy, CTA-pair GEMM
])
def test_static_scratch_forward_matches_oracle_and_workspace_forward(T, H, I, E, k, shared_I):
    import mixture_experts_layer_03_gb300 as moe
    lib = moe._lib
    x, ids, sc, w13, w2, w13s, w2s = _inputs(T, H, I, E, k, shared_I, seed=T + E)
    p = moe.make_problem(T, H, I, E, k, shared_I)
    assert moe.moe_workspace_bytes(p) <= moe.MOE_STATIC_SCRATCH_BYTES
    ws = moe.alloc_workspace(p)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    y_ws = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    st = lib.moe_forward(ctypes.byref(p), _p(x), _p(ids), _p(sc), _p(w13), _p(w2), _p(w13s),
                         _p(w2s), _p(y_ws), ws.ptr, ws.nbytes, stream)
    assert st == moe.MOE_OK, lib.moe_last_error()
    torch.cuda.synchronize()
    y_ref = oracle.forward(_np64(x), ids.cpu().numpy(), sc.cpu().numpy(), _np64(w13), _np64(w2),
                           _np64(w13s), _np64(w2s))
    bound = Y_TOL * np.abs(y_ref).max()
    for _ in range(2):   # two calls in a row: the scratch keeps the previous call's contents
        y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = lib.moe_forward_static(ctypes.byref(p), _p(x), _p(ids), _p(sc), _p(w13), _p(w2),
                                    _p(w13s), _p(w2s), _p(y), stream)
        assert st == moe.MOE_OK, lib.moe_last_error()
        flags = ctypes.c_int32(-1)
        st = lib.moe_static_read_device_status(stream, ctypes.byref(flags))
        assert st == moe.MOE_OK and flags.value == 0
        err = np.abs(y.cpu().double().numpy() - y_ref).max()
        assert err <= bound, f"max|y - y_ref| = {err:.4e} > {bound:.4e}"
        assert torch.equal(y.view(torch.int16), y_ws.view(torch.int16))


def test_static_scratch_reports_bad_ids():
    """An expert id outside [0, E) (made on the host) is skipped and flagged in the static
    scratch's status word; the read clears it, and the next clean call reports nothing."""
    import mixture_experts_layer_03_gb300 as moe
    lib = moe._lib
    T, H, I, E, k = 96, 256, 128, 8, 2
    x, ids, sc, w13, w2, _, _ = _inputs(T, H, I, E, k, 0, seed=5)
    bad = ids.clone()
    bad[7, 1] = E
    bad[40, 0] = -2
    p = moe.make_problem(T, H, I, E, k)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    y = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    st = lib.moe_forward_static(ctypes.byref(p), _p(x), _p(bad), _p(sc), _p(w13), _p(w2), None,
                                None, _p(y), stream)
    assert st == moe.MOE_OK, lib.moe_last_error()
    flags = ctypes.c_int32(0)
    st = lib.moe_static_read_device_status(stream, ctypes.byref(flags))
    assert st == moe.MOE_ERR_DEVICE_BAD_ID and flags.value & moe.MOE_DEVICE_FLAG_BAD_ID
    assert lib.moe_static_read_device_status(stream, None) == moe.MOE_OK   # the read cleared it
    # the skipped slots contribute nothing: the oracle with their scales set to 0
    sc0 = sc.cpu().numpy().copy()
    sc0[7, 1] = 0
    sc0[40, 0] = 0
    ids_ok = bad.cpu().numpy().copy()
    ids_ok[7, 1] = 0
    ids_ok[40, 0] = 0
    y_ref = oracle.forward(_np64(x), ids_ok, sc0, _np64(w13), _np64(w2))
    err = np.abs(y.cpu().double().numpy() - y_ref).max()
    assert err <= Y_TOL * np.abs(y_ref).max(), err
    st = lib.moe_forward_static(ctypes.byref(p), _p(x), _p(ids), _p(sc), _p(w13), _p(w2), None,
                                None, _p(y), stream)
    assert st == moe.MOE_OK
    assert lib.moe_static_read_device_status(stream, ctypes.byref(flags)) == moe.MOE_OK
    assert flags.value == 0


def test_static_scratch_rejects_problems_that_do_not_fit():
    import mixture_experts_layer_03_gb300 as moe
    p = moe.make_problem(T=4096, H=4096, I=14336, E=8, k=2)
    assert moe.moe_workspace_bytes(p) > moe.MOE_STATIC_SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: the size check comes first
    st = moe._lib.moe_forward_static(ctypes.byref(p), fake, fake, fake, fake, fake, None, None,
                                     fake, None)
    assert st == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    assert b"static scratch" in moe._lib.moe_last_error()

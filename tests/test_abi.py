"""CPU-side checks of the C ABI: the library builds, loads, exports every function
include/moe.h declares, and its host-only logic (envelope checks, workspace layout,
synchronous argument errors) behaves as documented. No GPU needed."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def moe():
    lib_path = os.path.join(ROOT, "mixture_experts_layer_03_gb300", "libmoe_gb300.so")
    if not os.path.exists(lib_path):
        if not (shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")):
            pytest.skip("library not built and nvcc unavailable")
        import __graft_entry__
        __graft_entry__.build()
    import mixture_experts_layer_03_gb300 as m
    return m


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(moe_[a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_step_calls():
    names = _declared_functions()
    for n in ("moe_route", "moe_forward", "moe_permute", "moe_fc1", "moe_fc2", "moe_fc1_fc2",
              "moe_finalize",
              "moe_can_implement", "moe_workspace_bytes", "moe_read_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(moe):
    lib = ctypes.CDLL(moe.LIB_PATH)
    for n in _declared_functions():
        assert hasattr(lib, n), n
    assert set(_declared_functions()) == set(moe.EXPORTED)
    assert moe._lib.moe_abi_version() == 1


def test_status_strings(moe):
    for s in range(8):
        assert moe._lib.moe_status_string(s).decode()
    assert moe._lib.moe_status_string(99).decode() == "unknown status"


@pytest.mark.parametrize("kw,reason", [
    (dict(T=64, H=128, I=256, E=8, k=2), 0),
    (dict(T=-1, H=128, I=256, E=8, k=2), 1),
    (dict(T=64, H=128, I=256, E=0, k=2), 2),
    (dict(T=64, H=128, I=256, E=257, k=2), 2),
    (dict(T=64, H=128, I=256, E=8, k=9), 3),
    (dict(T=64, H=100, I=256, E=8, k=2), 4),
    (dict(T=64, H=128, I=96, E=8, k=2), 5),
    (dict(T=64, H=128, I=256, E=8, k=2, shared_I=100), 6),
    (dict(T=4096, H=4096, I=14336, E=8, k=2), 0),
    (dict(T=512, H=7168, I=2048, E=256, k=8, shared_I=2048), 0),
])
def test_can_implement(moe, kw, reason):
    st, r = moe.moe_can_implement(moe.make_problem(**kw))
    assert r == reason
    assert (st == moe.MOE_OK) == (reason == 0)


def test_workspace_layout(moe):
    p = moe.make_problem(T=512, H=7168, I=2048, E=256, k=8, shared_I=2048)
    L = moe.moe_workspace_layout(p)
    P, R = 512 * 8, 512 * 8 + 512
    assert L["rows"] == R and L["groups"] == 257 and L["h_ld"] == 2048 and L["n_chunks"] == 4
    names = ["status", "counts", "starts", "offsets", "tile_off1", "tile_off2", "sched", "block_hist",
             "perm_src", "perm_inv", "x_perm", "h", "out_perm", "total"]
    offs = [L[n] for n in names]
    assert offs == sorted(offs) and all(o % 1024 == 0 for o in offs)
    assert L["x_perm"] >= L["perm_inv"] + 4 * P
    assert L["h"] - L["x_perm"] >= 2 * R * 7168
    assert L["out_perm"] - L["h"] >= 2 * R * 2048
    assert L["total"] - L["out_perm"] >= 2 * R * 7168
    assert moe.moe_workspace_bytes(p) == L["total"]
    assert moe.moe_workspace_bytes(moe.make_problem(T=1, H=100, I=64, E=1, k=1)) == 0
    # a wider shared expert widens h
    L2 = moe.moe_workspace_layout(moe.make_problem(T=10, H=128, I=64, E=4, k=2, shared_I=192))
    assert L2["h_ld"] == 192 and L2["groups"] == 5


def _route_params(moe, E, k, method, n_group=1, topk_group=1, rsf=1.0):
    return moe.MoeRouteParams(E, k, method, n_group, topk_group, rsf)


@pytest.mark.parametrize("E,k,method,ng,tg,ok", [
    (8, 2, 4, 1, 1, True), (8, 9, 4, 1, 1, False), (8, 9, 0, 1, 1, False), (4, 5, 1, 1, 1, False),
    (300, 2, 6, 1, 1, False), (8, 2, 3, 1, 1, True), (8, 2, 5, 1, 1, True),
    (256, 8, 5, 1, 1, True), (300, 8, 5, 1, 1, False), (16, 9, 3, 1, 1, False),
    (8, 2, 7, 1, 1, False), (8, 2, -1, 1, 1, False),   # no such method
    (256, 8, 2, 8, 4, True), (256, 8, 2, 7, 4, False), (256, 8, 2, 8, 9, False),
    (64, 8, 2, 1, 1, False),   # 64 experts in one group > 32 per group
    (8, 8, 2, 4, 2, False),    # k > topk_group * experts per group
    (8, 4, 2, 4, 2, True), (8, 2, 2, 8, 2, False),   # one expert per group: no top-2
    # vLLM grouped top-k: k / topk_group experts from each kept group
    (256, 8, 16, 8, 4, True), (32, 8, 16, 32, 8, True), (256, 8, 16, 1, 1, True),
    (256, 6, 16, 8, 4, False),   # 6 % 4 != 0
    (16, 8, 16, 8, 2, False),    # 4 per group > 2 experts per group
    (256, 8, 16, 64, 8, False),  # more than 32 groups
    (96, 4, 16, 5, 2, False),    # 96 % 5 != 0
])
def test_route_envelope_is_checked_on_the_host(moe, E, k, method, ng, tg, ok):
    """T = 0 enqueues nothing; an unsupported configuration is rejected synchronously."""
    p = _route_params(moe, E, k, method, ng, tg)
    st = moe._lib.moe_route(None, 0, None, ctypes.byref(p), None, None, None)
    assert (st == moe.MOE_OK) == ok, moe._lib.moe_last_error()
    if not ok:
        assert st == moe.MOE_ERR_UNSUPPORTED


def test_grouped_topk_softmax_is_refused_and_bias_rejected(moe):
    p = _route_params(moe, 256, 8, moe.MOE_ROUTE_GROUPED_TOPK_SOFTMAX, 8, 4)
    st = moe._lib.moe_route(None, 0, None, ctypes.byref(p), None, None, None)
    assert st == moe.MOE_ERR_UNSUPPORTED
    assert b"tie-breaking" in moe._lib.moe_last_error()
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: the bias check comes first
    p = _route_params(moe, 256, 8, moe.MOE_ROUTE_GROUPED_TOPK, 8, 4)
    st = moe._lib.moe_route(fake, 4, fake, ctypes.byref(p), fake, fake, None)
    assert st == moe.MOE_ERR_INVALID_ARG


def test_gate_route_host_errors(moe):
    lib = moe._lib
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: every call below fails on the host
    p = _route_params(moe, 8, 2, 4)
    # T = 0 is a no-op
    assert lib.moe_gate_route(None, None, 0, 128, 0, None, ctypes.byref(p), None, None, None, None,
                              None) == moe.MOE_OK
    # H not a multiple of 64, E too large, bad routing
    assert lib.moe_gate_route(fake, fake, 4, 100, 0, None, ctypes.byref(p), fake, fake, None, None,
                              None) == moe.MOE_ERR_UNSUPPORTED
    big = _route_params(moe, 300, 2, 4)
    assert lib.moe_gate_route(fake, fake, 4, 128, 0, None, ctypes.byref(big), fake, fake, None,
                              None, None) == moe.MOE_ERR_UNSUPPORTED
    soft = _route_params(moe, 256, 8, moe.MOE_ROUTE_GROUPED_TOPK_SOFTMAX, 8, 4)
    assert lib.moe_gate_route(fake, fake, 4, 128, 0, None, ctypes.byref(soft), fake, fake, None,
                              None, None) == moe.MOE_ERR_UNSUPPORTED
    # missing outputs, misaligned pointers, a shared gate row without its output
    assert lib.moe_gate_route(fake, fake, 4, 128, 0, None, ctypes.byref(p), None, fake, None, None,
                              None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_gate_route(ctypes.c_void_p((1 << 20) + 4), fake, 4, 128, 0, None,
                              ctypes.byref(p), fake, fake, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_gate_route(fake, fake, 4, 128, 1, None, ctypes.byref(p), fake, fake, None, None,
                              None) == moe.MOE_ERR_INVALID_ARG
    gt = _route_params(moe, 256, 8, moe.MOE_ROUTE_GROUPED_TOPK, 8, 4)
    assert lib.moe_gate_route(fake, fake, 4, 128, 0, fake, ctypes.byref(gt), fake, fake, None, None,
                              None) == moe.MOE_ERR_INVALID_ARG


def test_forward_host_errors(moe):
    p = moe.make_problem(T=16, H=128, I=64, E=4, k=2)
    n = moe.moe_workspace_bytes(p)
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: every call below fails on the host
    lib = moe._lib
    # NULL workspace
    assert lib.moe_forward(ctypes.byref(p), fake, fake, fake, fake, fake, None, None, fake,
                           None, n, None) == moe.MOE_ERR_INVALID_ARG
    # misaligned workspace
    assert lib.moe_forward(ctypes.byref(p), fake, fake, fake, fake, fake, None, None, fake,
                           ctypes.c_void_p((1 << 20) + 256), n, None) == moe.MOE_ERR_INVALID_ARG
    # workspace too small
    assert lib.moe_forward(ctypes.byref(p), fake, fake, fake, fake, fake, None, None, fake,
                           fake, n - 1, None) == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    # misaligned tensor
    assert lib.moe_forward(ctypes.byref(p), ctypes.c_void_p((1 << 20) + 2), fake, fake, fake, fake,
                           None, None, fake, fake, n, None) == moe.MOE_ERR_INVALID_ARG
    # unsupported shape
    bad = moe.make_problem(T=16, H=96, I=64, E=4, k=2)
    assert lib.moe_forward(ctypes.byref(bad), fake, fake, fake, fake, fake, None, None, fake,
                           fake, n, None) == moe.MOE_ERR_UNSUPPORTED
    # shared expert requested but its weights missing
    ps = moe.make_problem(T=16, H=128, I=64, E=4, k=2, shared_I=64)
    ns = moe.moe_workspace_bytes(ps)
    assert lib.moe_forward(ctypes.byref(ps), fake, fake, fake, fake, fake, None, None, fake,
                           fake, ns, None) == moe.MOE_ERR_INVALID_ARG
    # T = 0 is a no-op, even with NULL pointers
    p0 = moe.make_problem(T=0, H=128, I=64, E=4, k=2)
    assert lib.moe_forward(ctypes.byref(p0), None, None, None, None, None, None, None, None,
                           None, 0, None) == moe.MOE_OK
    for fn in (lib.moe_permute,):
        assert fn(ctypes.byref(p0), None, None, None, 0, None) == moe.MOE_OK
    assert lib.moe_cast_f32_to_bf16(None, None, -1, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_cast_f32_to_bf16(None, None, 0, None) == moe.MOE_OK
    assert lib.moe_read_device_status(None, None, None) == moe.MOE_ERR_INVALID_ARG
    # the failure-path self-test checks its workspace pointer on the host
    assert lib.moe_selftest_wait(None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_wait(ctypes.c_void_p(8), None) == moe.MOE_ERR_INVALID_ARG

"""Python binding of the GB300 MoE layer forward library (libmoe_gb300.so).

Argument marshalling only: every step runs in the library's CUDA kernels. PyTorch
provides device memory and streams. The names mirror the C ABI in include/moe.h.
Importing this module fails loudly when the compiled library is missing; there is
no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

MOE_ROUTE_DEFAULT = 0
MOE_ROUTE_RENORMALIZE = 1
MOE_ROUTE_DEEPSEEKV3 = 2
MOE_ROUTE_LLAMA4 = 3
MOE_ROUTE_RENORMALIZE_NAIVE = 4
MOE_ROUTE_MINIMAX2 = 5
MOE_ROUTE_SIGMOID_RENORM = 6
MOE_ROUTE_GROUPED_TOPK = 16
MOE_ROUTE_GROUPED_TOPK_SOFTMAX = 17

MOE_REASON_DEGENERATE = 10

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE_TOO_SMALL = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_BAD_ID = 5
MOE_ERR_DEVICE_TIMEOUT = 6
MOE_ERR_NOT_IMPLEMENTED = 7

MOE_DEVICE_FLAG_BAD_ID = 1
MOE_DEVICE_FLAG_TIMEOUT = 2


class MoeProblem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("shared_I", ctypes.c_int32)]


class MoeRouteParams(ctypes.Structure):
    _fields_ = [("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("method", ctypes.c_int32), ("n_group", ctypes.c_int32),
                ("topk_group", ctypes.c_int32), ("routed_scaling_factor", ctypes.c_float)]


class MoeWsLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("status", "counts", "starts", "offsets", "tile_off1", "tile_off2", "sched", "block_hist",
                 "perm_src", "perm_inv", "x_perm", "h", "out_perm", "total")] + \
               [("rows", ctypes.c_int64), ("groups", ctypes.c_int32), ("n_chunks", ctypes.c_int32),
                ("h_ld", ctypes.c_int32), ("reserved", ctypes.c_int32)]


# Every exported symbol of include/moe.h, with its ctypes signature.
_P = ctypes.c_void_p
_SIGS = {
    "moe_abi_version": (ctypes.c_int32, []),
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_last_error": (ctypes.c_char_p, []),
    "moe_route": (ctypes.c_int, [_P, ctypes.c_int64, _P, ctypes.POINTER(MoeRouteParams), _P, _P, _P]),
    "moe_can_implement": (ctypes.c_int, [ctypes.POINTER(MoeProblem), ctypes.POINTER(ctypes.c_int32)]),
    "moe_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(MoeProblem)]),
    "moe_workspace_layout": (ctypes.c_int, [ctypes.POINTER(MoeProblem), ctypes.POINTER(MoeWsLayout)]),
    "moe_forward": (ctypes.c_int, [ctypes.POINTER(MoeProblem), _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                   ctypes.c_size_t, _P]),
    "moe_forward_static": (ctypes.c_int, [ctypes.POINTER(MoeProblem), _P, _P, _P, _P, _P, _P, _P,
                                          _P, _P]),
    "moe_forward_partial": (ctypes.c_int, [ctypes.POINTER(MoeProblem), ctypes.c_int32,
                                           ctypes.c_int32, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                           _P, ctypes.c_size_t, _P]),
    "moe_gate": (ctypes.c_int, [_P, _P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                ctypes.c_int32, _P, _P, _P]),
    "moe_gate_route": (ctypes.c_int, [_P, _P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _P,
                                      ctypes.POINTER(MoeRouteParams), _P, _P, _P, _P, _P]),
    "moe_permute": (ctypes.c_int, [ctypes.POINTER(MoeProblem), _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_fc1": (ctypes.c_int, [ctypes.POINTER(MoeProblem), _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_fc2": (ctypes.c_int, [ctypes.POINTER(MoeProblem), _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_fc1_fc2": (ctypes.c_int, [ctypes.POINTER(MoeProblem), _P, _P, _P, _P, _P, ctypes.c_size_t,
                                   _P]),
    "moe_finalize": (ctypes.c_int, [ctypes.POINTER(MoeProblem), _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_read_device_status": (ctypes.c_int, [_P, _P, ctypes.POINTER(ctypes.c_int32)]),
    "moe_static_read_device_status": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int32)]),
    "moe_selftest_wait": (ctypes.c_int, [_P, _P]),
    "moe_cast_f32_to_bf16": (ctypes.c_int, [_P, _P, ctypes.c_int64, _P]),
}
EXPORTED = tuple(_SIGS)


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the compiled library and attach the C signatures."""
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = load_library()


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = _lib.moe_status_string(status).decode()
        detail = _lib.moe_last_error().decode()
        super().__init__(f"{where}: {msg} ({status}) {detail}")
        self.status = status


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _cuda(t: torch.Tensor, name: str, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def make_problem(T, H, I, E, k, shared_I=0) -> MoeProblem:
    return MoeProblem(int(T), int(H), int(I), int(E), int(k), int(shared_I))


def moe_can_implement(problem: MoeProblem):
    reason = ctypes.c_int32(0)
    st = _lib.moe_can_implement(ctypes.byref(problem), ctypes.byref(reason))
    return st, reason.value


def moe_workspace_bytes(problem: MoeProblem) -> int:
    return int(_lib.moe_workspace_bytes(ctypes.byref(problem)))


def moe_workspace_layout(problem: MoeProblem) -> dict:
    L = MoeWsLayout()
    _check(_lib.moe_workspace_layout(ctypes.byref(problem), ctypes.byref(L)), "moe_workspace_layout")
    return {n: getattr(L, n) for n, _ in MoeWsLayout._fields_}


@dataclass
class Workspace:
    """Caller-owned device workspace (a torch byte buffer, 1024-byte aligned view)."""
    problem: MoeProblem
    buf: torch.Tensor
    base: int           # byte offset of the aligned start inside buf
    nbytes: int
    layout: dict

    @property
    def ptr(self) -> ctypes.c_void_p:
        return ctypes.c_void_p(self.buf.data_ptr() + self.base)

    def region(self, name: str, count: int, dtype: torch.dtype) -> torch.Tensor:
        off = self.base + self.layout[name]
        nbytes = count * torch.empty((), dtype=dtype).element_size()
        return self.buf[off:off + nbytes].view(dtype)


def alloc_workspace(problem: MoeProblem, device="cuda") -> Workspace:
    n = moe_workspace_bytes(problem)
    if n == 0:
        raise MoeError(MOE_ERR_UNSUPPORTED, "moe_workspace_bytes")
    buf = torch.empty(n + 1024, dtype=torch.uint8, device=device)
    base = (-buf.data_ptr()) % 1024
    return Workspace(problem, buf, base, n, moe_workspace_layout(problem))


def moe_route(logits: torch.Tensor, method: int, top_k: int, bias: Optional[torch.Tensor] = None,
              n_group: int = 1, topk_group: int = 1, routed_scaling_factor: float = 1.0,
              ids: Optional[torch.Tensor] = None, scales: Optional[torch.Tensor] = None,
              stream=None):
    """Routing: logits fp32 [T, E] -> (ids int32 [T, k], scales fp32 [T, k])."""
    _cuda(logits, "logits", torch.float32)
    T, E = logits.shape
    if bias is not None:
        _cuda(bias, "bias", torch.float32)
    if ids is None:
        ids = torch.empty((T, top_k), dtype=torch.int32, device=logits.device)
    if scales is None:
        scales = torch.empty((T, top_k), dtype=torch.float32, device=logits.device)
    p = MoeRouteParams(E, top_k, method, n_group, topk_group, routed_scaling_factor)
    _check(_lib.moe_route(_ptr(logits), T, _ptr(bias), ctypes.byref(p), _ptr(ids), _ptr(scales),
                          _stream(stream)), "moe_route")
    return ids, scales


def _problem_for(x, ids, w13, w2, w13_s):
    T, H = x.shape
    k = ids.shape[1]
    E, twoI, _ = w13.shape
    return make_problem(T, H, twoI // 2, E, k, 0 if w13_s is None else w13_s.shape[0] // 2)


def moe_forward(x, ids, scales, w13, w2, w13_s=None, w2_s=None, y=None,
                workspace: Optional[Workspace] = None, stream=None):
    """Steps 2-5: permute, FC1+SwiGLU, FC2, finalize. Returns y bf16 [T, H]."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(ids, "ids", torch.int32)
    _cuda(scales, "scales", torch.float32)
    _cuda(w13, "w13", torch.bfloat16)
    _cuda(w2, "w2", torch.bfloat16)
    p = _problem_for(x, ids, w13, w2, w13_s)
    if workspace is None:
        workspace = alloc_workspace(p, x.device)
    if y is None:
        y = torch.empty_like(x)
    _check(_lib.moe_forward(ctypes.byref(p), _ptr(x), _ptr(ids), _ptr(scales), _ptr(w13), _ptr(w2),
                            _ptr(w13_s), _ptr(w2_s), _ptr(y), workspace.ptr, workspace.nbytes,
                            _stream(stream)), "moe_forward")
    return y


def moe_forward_partial(x, ids, scales, w13_local, w2_local, e_lo: int, e_hi: int, num_experts: int,
                        w13_s=None, w2_s=None, shared_gate=None, y=None,
                        workspace: Optional[Workspace] = None, stream=None):
    """moe_forward over the experts [e_lo, e_hi) of num_experts only (the expert-parallel
    seam): slots routed elsewhere contribute 0. w13_local / w2_local hold those experts'
    weights, [e_hi - e_lo, 2I, H] / [e_hi - e_lo, H, I]. shared_gate: fp32 [T] logits that
    weight the shared expert by their sigmoid (None: weight 1). Returns y bf16 [T, H]."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(ids, "ids", torch.int32)
    _cuda(scales, "scales", torch.float32)
    _cuda(w13_local, "w13_local", torch.bfloat16)
    _cuda(w2_local, "w2_local", torch.bfloat16)
    T, H = x.shape
    k = ids.shape[1]
    I = w2_local.shape[2]
    shared_I = 0 if w13_s is None else w13_s.shape[0] // 2
    p = make_problem(T, H, I, num_experts, k, shared_I)
    if workspace is None:
        workspace = alloc_workspace(p, x.device)
    if y is None:
        y = torch.empty_like(x)
    if shared_gate is not None:
        _cuda(shared_gate, "shared_gate", torch.float32)
    _check(_lib.moe_forward_partial(ctypes.byref(p), int(e_lo), int(e_hi), _ptr(x), _ptr(ids),
                                    _ptr(scales), _ptr(w13_local), _ptr(w2_local), _ptr(w13_s),
                                    _ptr(w2_s), _ptr(shared_gate), _ptr(y), workspace.ptr,
                                    workspace.nbytes, _stream(stream)), "moe_forward_partial")
    return y


def moe_gate(x, wg, num_experts: int, routed_logits=None, shared_logits=None, stream=None):
    """Router gate: x bf16 [T, H] . wg bf16 [E (+1), H]^T -> (routed logits fp32 [T, E],
    shared-expert gate logits fp32 [T] or None). A wg with E + 1 rows carries the fused
    shared-expert gate in its last row."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(wg, "wg", torch.bfloat16)
    T, H = x.shape
    E = int(num_experts)
    n_shared = wg.shape[0] - E
    if n_shared not in (0, 1) or wg.shape[1] != H:
        raise ValueError(f"wg must be [{E} or {E + 1}, {H}], got {tuple(wg.shape)}")
    if routed_logits is None:
        routed_logits = torch.empty((T, E), dtype=torch.float32, device=x.device)
    if n_shared and shared_logits is None:
        shared_logits = torch.empty((T,), dtype=torch.float32, device=x.device)
    _check(_lib.moe_gate(_ptr(x), _ptr(wg), T, H, E, n_shared, _ptr(routed_logits),
                         _ptr(shared_logits) if n_shared else None, _stream(stream)), "moe_gate")
    return routed_logits, (shared_logits if n_shared else None)


def moe_gate_route(x, wg, method: int, top_k: int, num_experts: int,
                   bias: Optional[torch.Tensor] = None, n_group: int = 1, topk_group: int = 1,
                   routed_scaling_factor: float = 1.0, ids=None, scales=None,
                   routed_logits=None, shared_logits=None, want_logits: bool = False,
                   stream=None):
    """Router gate and routing in one launch: x bf16 [T, H], wg bf16 [E (+1), H] ->
    (ids int32 [T, k], scales fp32 [T, k], routed logits fp32 [T, E] or None, shared-expert
    gate logits fp32 [T] or None). The routed logits are written only when want_logits is
    set or routed_logits is passed."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(wg, "wg", torch.bfloat16)
    T, H = x.shape
    E = int(num_experts)
    n_shared = wg.shape[0] - E
    if n_shared not in (0, 1) or wg.shape[1] != H:
        raise ValueError(f"wg must be [{E} or {E + 1}, {H}], got {tuple(wg.shape)}")
    if bias is not None:
        _cuda(bias, "bias", torch.float32)
    if ids is None:
        ids = torch.empty((T, top_k), dtype=torch.int32, device=x.device)
    if scales is None:
        scales = torch.empty((T, top_k), dtype=torch.float32, device=x.device)
    if want_logits and routed_logits is None:
        routed_logits = torch.empty((T, E), dtype=torch.float32, device=x.device)
    if n_shared and shared_logits is None:
        shared_logits = torch.empty((T,), dtype=torch.float32, device=x.device)
    p = MoeRouteParams(E, top_k, method, n_group, topk_group, routed_scaling_factor)
    _check(_lib.moe_gate_route(_ptr(x), _ptr(wg), T, H, n_shared, _ptr(bias), ctypes.byref(p),
                               _ptr(ids), _ptr(scales), _ptr(routed_logits),
                               _ptr(shared_logits) if n_shared else None, _stream(stream)),
           "moe_gate_route")
    return ids, scales, routed_logits, (shared_logits if n_shared else None)


MOE_STATIC_SCRATCH_BYTES = 32 << 20


def moe_forward_static(x, ids, scales, w13, w2, w13_s=None, w2_s=None, y=None, stream=None):
    """moe_forward with the library's built-in scratch instead of a caller workspace.

    For callers that cannot allocate device memory (a plugin whose host engine owns all
    device allocations, or a loop that must not call cudaMalloc). Problems whose workspace
    exceeds MOE_STATIC_SCRATCH_BYTES are rejected. All calls on a GPU share one scratch
    array, so calls that overlap on the GPU race; the first call on a device sets the
    array up and should come before any stream capture. ``y`` is allocated here (by
    torch) only when the caller does not pass it.
    """
    _cuda(x, "x", torch.bfloat16)
    _cuda(ids, "ids", torch.int32)
    _cuda(scales, "scales", torch.float32)
    _cuda(w13, "w13", torch.bfloat16)
    _cuda(w2, "w2", torch.bfloat16)
    p = _problem_for(x, ids, w13, w2, w13_s)
    if y is None:
        y = torch.empty_like(x)
    _check(_lib.moe_forward_static(ctypes.byref(p), _ptr(x), _ptr(ids), _ptr(scales), _ptr(w13),
                                   _ptr(w2), _ptr(w13_s), _ptr(w2_s), _ptr(y), _stream(stream)),
           "moe_forward_static")
    return y


def moe_permute(problem, x, ids, workspace: Workspace, stream=None):
    _check(_lib.moe_permute(ctypes.byref(problem), _ptr(x), _ptr(ids), workspace.ptr,
                            workspace.nbytes, _stream(stream)), "moe_permute")


def moe_fc1(problem, w13, w13_s, workspace: Workspace, stream=None):
    _check(_lib.moe_fc1(ctypes.byref(problem), _ptr(w13), _ptr(w13_s), workspace.ptr,
                        workspace.nbytes, _stream(stream)), "moe_fc1")


def moe_fc2(problem, w2, w2_s, workspace: Workspace, stream=None):
    _check(_lib.moe_fc2(ctypes.byref(problem), _ptr(w2), _ptr(w2_s), workspace.ptr,
                        workspace.nbytes, _stream(stream)), "moe_fc2")


def moe_fc1_fc2(problem, w13, w13_s, w2, w2_s, workspace: Workspace, stream=None):
    _check(_lib.moe_fc1_fc2(ctypes.byref(problem), _ptr(w13), _ptr(w13_s), _ptr(w2), _ptr(w2_s),
                            workspace.ptr, workspace.nbytes, _stream(stream)), "moe_fc1_fc2")


def moe_finalize(problem, scales, y, workspace: Workspace, stream=None):
    _check(_lib.moe_finalize(ctypes.byref(problem), _ptr(scales), _ptr(y), workspace.ptr,
                             workspace.nbytes, _stream(stream)), "moe_finalize")


def moe_read_device_status(workspace: Workspace, stream=None):
    """Synchronise, read and clear the device status word. Returns (status, flags)."""
    flags = ctypes.c_int32(0)
    st = _lib.moe_read_device_status(workspace.ptr, _stream(stream), ctypes.byref(flags))
    return st, flags.value


def moe_static_read_device_status(stream=None):
    """Synchronise, read and clear moe_forward_static's status word on the current device.
    Returns (status, flags)."""
    flags = ctypes.c_int32(0)
    st = _lib.moe_static_read_device_status(_stream(stream), ctypes.byref(flags))
    return st, flags.value


def moe_selftest_wait(workspace: Workspace, stream=None):
    """Enqueue the device failure-path self-test on ``workspace``'s status words: a
    bounded wait that runs out after about 2 s and reports MOE_DEVICE_FLAG_TIMEOUT."""
    _check(_lib.moe_selftest_wait(workspace.ptr, _stream(stream)), "moe_selftest_wait")


def moe_cast_f32_to_bf16(t: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None):
    _cuda(t, "input", torch.float32)
    if out is None:
        out = torch.empty(t.shape, dtype=torch.bfloat16, device=t.device)
    _check(_lib.moe_cast_f32_to_bf16(_ptr(t), _ptr(out), t.numel(), _stream(stream)),
           "moe_cast_f32_to_bf16")
    return out


__all__ = [n for n in dir() if n.startswith(("moe_", "MOE_", "Moe"))] + [
    "make_problem", "alloc_workspace", "Workspace", "load_library", "EXPORTED", "LIB_PATH"]

"""Seeded synthetic inputs for the MoE layer forward.

This module holds no arithmetic of the method: only the shapes, value
distributions and draw order of the workloads. Both sides of every parity
check (the CPU oracle and the CUDA path) consume the tensors made here.

Recipe (all draws from one ``torch.Generator`` seeded with ``seed``, on the
device the caller names, in this fixed order):

1. ``logits`` [T, E] fp32 ~ N(0, 1) (plus a per-expert Zipf bias for the
   skewed workload, see ``zipf_logit_bias``);
2. ``bias`` [E] fp32 ~ N(0, bias_std) (the biased-key routings, DeepSeek-V3 and MiniMax2);
3. ``x`` [T, H] ~ N(0, 1);
4. ``w13`` [E, 2I, H], expert by expert, ~ N(0, std = H^-1/2);
5. ``w2`` [E, H, I], expert by expert, ~ N(0, std = I^-1/2);
6. shared expert ``w13_s`` [2Is, H] ~ N(0, H^-1/2), ``w2_s`` [H, Is] ~ N(0, Is^-1/2).

Every tensor is drawn in fp32 and then rounded to bf16 (round to nearest
even) where the workload is bf16; the tiny workload keeps fp32 tensors.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

# Routing method codes (the RoutingMethodType enum values of the TensorRT-LLM
# MoE page, section "路由方法枚举").
DEFAULT = 0
RENORMALIZE = 1
DEEPSEEKV3 = 2
LLAMA4 = 3
RENORMALIZE_NAIVE = 4
MINIMAX2 = 5
SIGMOID_RENORM = 6
# vLLM's GroupedTopKRouter with sigmoid scoring (vLLM MoE page, section "GroupedTopKRouter");
# a code outside the RoutingMethodType range.
GROUPED_TOPK = 16


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    method: int
    n_group: int = 1
    topk_group: int = 1
    rsf: float = 1.0
    shared_I: int = 0
    bias_std: float = 0.0
    zipf_s: float = 0.0          # >0: add 3*ln(Zipf rank weight) to each expert's logits
    in_dtype: str = "bf16"       # "f32" for the tiny workload

    @property
    def P(self) -> int:
        return self.T * self.k

    def describe(self) -> str:
        s = f"{self.name}: T={self.T} H={self.H} I={self.I} E={self.E} k={self.k} method={self.method}"
        if self.n_group > 1:
            s += f" n_group={self.n_group} topk_group={self.topk_group}"
        if self.rsf != 1.0:
            s += f" rsf={self.rsf}"
        if self.shared_I:
            s += f" shared_I={self.shared_I}"
        return s


WORKLOADS = {
    "tiny": Workload("tiny", T=64, H=128, I=256, E=8, k=2, method=RENORMALIZE_NAIVE, in_dtype="f32"),
    "mixtral_prefill": Workload("mixtral_prefill", T=4096, H=4096, I=14336, E=8, k=2,
                                method=RENORMALIZE_NAIVE),
    "qwen3_decode": Workload("qwen3_decode", T=64, H=2048, I=768, E=128, k=8,
                             method=RENORMALIZE_NAIVE),
    "dsv3_layer": Workload("dsv3_layer", T=512, H=7168, I=2048, E=256, k=8, method=DEEPSEEKV3,
                           n_group=8, topk_group=4, rsf=2.5, shared_I=2048, bias_std=0.1),
    "skewed": Workload("skewed", T=8192, H=4096, I=1536, E=64, k=4, method=SIGMOID_RENORM,
                       zipf_s=1.2),
    # Shapes of the two routing methods the TensorRT-LLM page names by model (Llama4:
    # "Top1 -> Sigmoid"; MiniMaxM2: sigmoid + bias -> top-k -> renormalise without bias),
    # taken from those models' published layer sizes.
    "llama4_scout": Workload("llama4_scout", T=2048, H=5120, I=8192, E=16, k=1, method=LLAMA4,
                             shared_I=8192),
    "minimax_m2": Workload("minimax_m2", T=4096, H=3072, I=1536, E=256, k=8, method=MINIMAX2,
                           bias_std=0.1),
}
ORDER = ["tiny", "mixtral_prefill", "qwen3_decode", "dsv3_layer", "skewed", "llama4_scout",
         "minimax_m2"]


def zipf_logit_bias(E: int, s: float) -> torch.Tensor:
    """3*ln(w_r) for Zipf rank weights w_r = r^-s / sum_r' r'^-s, rank r = expert index + 1."""
    r = torch.arange(1, E + 1, dtype=torch.float64)
    w = r.pow(-s)
    w = w / w.sum()
    return (3.0 * torch.log(w)).to(torch.float32)


def _randn(shape, gen, device, std=1.0):
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def make_inputs(w: Workload, device="cpu", seed: int = 0, weights: bool = True,
                T: Optional[int] = None):
    """Draw one workload's inputs. Returns a dict of tensors on ``device``.

    ``T`` overrides the token count (the draw order is unchanged).
    ``weights=False`` skips the expert weights (routing-only checks).
    """
    T = w.T if T is None else T
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    wdt = torch.float32 if w.in_dtype == "f32" else torch.bfloat16
    out = {}
    logits = _randn((T, w.E), gen, device)
    if w.zipf_s > 0:
        logits += zipf_logit_bias(w.E, w.zipf_s).to(device)
    out["logits"] = logits
    out["bias"] = _randn((w.E,), gen, device, w.bias_std) if w.bias_std > 0 else None
    out["x"] = _randn((T, w.H), gen, device).to(wdt)
    if not weights:
        return out
    w13 = torch.empty((w.E, 2 * w.I, w.H), dtype=wdt, device=device)
    for e in range(w.E):
        w13[e] = _randn((2 * w.I, w.H), gen, device, w.H ** -0.5).to(wdt)
    w2 = torch.empty((w.E, w.H, w.I), dtype=wdt, device=device)
    for e in range(w.E):
        w2[e] = _randn((w.H, w.I), gen, device, w.I ** -0.5).to(wdt)
    out["w13"], out["w2"] = w13, w2
    if w.shared_I:
        out["w13_s"] = _randn((2 * w.shared_I, w.H), gen, device, w.H ** -0.5).to(wdt)
        out["w2_s"] = _randn((w.H, w.shared_I), gen, device, w.shared_I ** -0.5).to(wdt)
    else:
        out["w13_s"] = out["w2_s"] = None
    return out


def small_case(name, T, H, I, E, k, method=RENORMALIZE_NAIVE, **kw) -> Workload:
    """A reduced-size workload for parity tests (same distributions)."""
    return Workload(name, T=T, H=H, I=I, E=E, k=k, method=method, **kw)


def flops(w: Workload) -> float:
    """Algorithmic FLOPs of the layer: 2*P*3*H*I (+ 2*T*3*H*Is for the shared expert)."""
    return 2.0 * w.P * 3 * w.H * w.I + 2.0 * w.T * 3 * w.H * w.shared_I


def min_bytes(w: Workload, n_active: int) -> float:
    """Algorithmic bytes: active experts' weights, shared weights, x, y, logits, ids, scales."""
    wb = 2  # bf16 weights and activations on the device path
    return (n_active * 3 * w.H * w.I * wb + 3 * w.H * w.shared_I * wb
            + 2 * w.T * w.H * wb + w.T * w.E * 4 + w.T * w.k * 8)


def pipeline_bytes(w: Workload, n_active: int) -> float:
    """What the permuted pipeline moves beyond `min_bytes`: x rows read and written into
    x_perm and read back by FC1, h written by FC1 and read by FC2, out_perm written by FC2
    and read by finalize, for the P routed rows (and the T shared-expert rows). A
    diagnostic beside the roofline, which counts `min_bytes` only."""
    wb = 2
    rows_r, rows_s = w.P, (w.T if w.shared_I else 0)
    return (min_bytes(w, n_active) + 5 * (rows_r + rows_s) * w.H * wb
            + 2 * (rows_r * w.I + rows_s * w.shared_I) * wb)


__all__ = ["Workload", "WORKLOADS", "ORDER", "make_inputs", "small_case", "zipf_logit_bias",
           "flops", "min_bytes", "pipeline_bytes", "DEFAULT", "RENORMALIZE", "DEEPSEEKV3", "LLAMA4",
           "RENORMALIZE_NAIVE", "MINIMAX2", "SIGMOID_RENORM", "GROUPED_TOPK"]

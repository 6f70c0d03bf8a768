"""CPU oracle for the MoE layer forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline
leg and its ``--impl reference`` arm) may import this module. The product path
(the C-ABI library and its Python binding) never calls it, and it shares no
code, table or helper with that path.

Plain, slow, obviously correct: numpy in float64, one step per definition,
no blocking or fusion. Sources (titles of the pages that define the method):

* [TRT] "TensorRT-LLM 源码完全拆解(十三): MoE 层前向执行——路由、Fused Kernel 与专家并行的三段拼装"
* [VLLM] "vLLM 源码完全拆解(八): MoE 层的前向执行"
* [GG] "从 Dense GEMM 到 TP MoE 的演进逻辑" (gsyq.cn news 428989), a GroupedGEMM / TP-MoE article

The layer computes (TRT, section "MoE 在推理侧到底特殊在哪里", the MoE formula)

    y = sum_{i in TopK(x)} g_i(x) * E_i(x)  (+ shared expert, TRT layer-structure figure)

with E_i a SwiGLU FFN. Readings taken where the pages are silent:

* Selection for the softmax/sigmoid methods is top-k of the raw fp32 logit
  (softmax and sigmoid are strictly increasing, so the chosen set and its order
  are those of the scores); ties go to the lowest expert index.
* Llama4 ("Top1 -> Sigmoid"): the top-k experts by logit (k = 1 in the model the
  name refers to), each weighted by the sigmoid of its own logit, not renormalised.
* MiniMaxM2 ("Sigmoid -> RoutingBiasAdd -> TopK -> Renormalize(without bias)"): the
  DeepSeek-V3 key below without groups, weights = unbiased sigmoid / their sum (no
  epsilon and no scaling factor: the pages name neither for this method).
* DeepSeek-V3 selection key: kappa_e = fl32(fl32(sigmoid64(l_e)) + b_e), i.e.
  the sigmoid in float64 rounded once to fp32, then an IEEE fp32 add of the
  bias. Group score = fl32(top1 + top2 of kappa within the group). Ties: lowest
  group index, then lowest expert index.
* vLLM GroupedTopKRouter (VLLM, section "GroupedTopKRouter：分组的专家选择"), sigmoid
  scoring: score s_e = sigmoid(l_e) in float64; selection key fl32(s_e), the score rounded
  once to fp32; group score = the sum of the group's keys added in fp32 in expert order;
  keep the topk_group best groups, then the k / topk_group best experts inside each of
  them; weights = s_sel / sum(s_sel) * routed_scaling_factor. With softmax scoring the
  group score is the sum of a softmax taken inside the group, 1 for every group, so the
  group choice would rest on tie-breaking alone; that form is refused.
* Output slots are listed by descending selection key.
* SwiGLU: the first I rows of w13[e] are the gate projection (w1), the next I
  rows the up projection (w3): h = silu(gate) * up, silu(z) = z / (1 + e^-z).
* The shared expert enters with weight 1 (the routed scaling factor is already
  inside the routed scales).
* Non-finite logits count as -inf for selection and for the normalisers.
"""
from __future__ import annotations

import numpy as np

DEFAULT = 0
RENORMALIZE = 1
DEEPSEEKV3 = 2
LLAMA4 = 3
RENORMALIZE_NAIVE = 4
MINIMAX2 = 5
SIGMOID_RENORM = 6

# vLLM's GroupedTopKRouter, by its scoring function. The codes lie outside the range of
# TensorRT-LLM's RoutingMethodType (0-8).
GROUPED_TOPK = 16
GROUPED_TOPK_SOFTMAX = 17

METHODS = (DEFAULT, RENORMALIZE, DEEPSEEKV3, LLAMA4, RENORMALIZE_NAIVE, MINIMAX2, SIGMOID_RENORM,
           GROUPED_TOPK)


# --------------------------------------------------------------------------- routing

def topk_desc(keys: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest keys per row, largest first, ties -> lowest index.

    A stable sort of the negated keys keeps equal keys in ascending index order.
    """
    return np.argsort(-keys, axis=-1, kind="stable")[..., :k]


def _selection_logits(logits32: np.ndarray) -> np.ndarray:
    return np.where(np.isfinite(logits32), logits32, np.float32(-np.inf)).astype(np.float32)


def softmax64(l: np.ndarray) -> np.ndarray:
    """Row softmax in float64; -inf entries get probability 0."""
    m = np.max(l, axis=-1, keepdims=True)
    z = np.exp(l - m)
    return z / np.sum(z, axis=-1, keepdims=True)


def sigmoid64(l: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-l))


def deepseek_keys(logits32: np.ndarray, bias32: np.ndarray):
    """(unbiased sigmoid scores in float64, fp32 selection keys kappa).

    TRT, section "DeepSeek-V3 的 noaux_tc:分组路由的算术": scores = sigmoid(logits),
    scores_with_bias = scores + e_score_correction_bias; the bias only decides who is
    chosen, the weights use the unbiased scores.
    """
    l = _selection_logits(logits32)
    s64 = sigmoid64(l.astype(np.float64))
    kappa = (s64.astype(np.float32) + bias32.astype(np.float32)).astype(np.float32)
    return s64, kappa


def group_select(kappa: np.ndarray, n_group: int, topk_group: int):
    """Chosen groups per token (group-score descending) and the group scores.

    TRT noaux_tc section: group score = sum of the top-2 biased scores inside the
    group; keep the topk_group best groups.
    """
    T, E = kappa.shape
    epg = E // n_group
    g = kappa.reshape(T, n_group, epg)
    top2 = -np.sort(-g, axis=-1)[..., :2]
    gscore = (top2[..., 0] + top2[..., 1]).astype(np.float32)
    groups = topk_desc(gscore, topk_group)
    return groups, gscore


def group_totals_fp32(keys: np.ndarray, n_group: int) -> np.ndarray:
    """Per-group sums of fp32 keys [T, E] -> [T, n_group], added in fp32 in expert order
    (((k0 + k1) + k2) + ...), each addition rounded to fp32."""
    T, E = keys.shape
    g = np.asarray(keys, np.float32).reshape(T, n_group, E // n_group)
    acc = g[..., 0].copy()
    for j in range(1, g.shape[-1]):
        acc = (acc + g[..., j]).astype(np.float32)
    return acc


def grouped_topk(logits32: np.ndarray, top_k: int, n_group: int, topk_group: int,
                 routed_scaling_factor: float = 1.0, scoring: str = "sigmoid"):
    """vLLM GroupedTopKRouter._select_experts, in the order VLLM lists its steps:

    1. view the logits as [T, n_group, experts_per_group];
    2. score inside each group (sigmoid here: s = sigmoid(l) in float64, key = fl32(s));
    3. group score = sum of the group's scores (fp32 keys added in expert order), keep the
       topk_group best groups (ties: lower group index);
    4. inside each kept group, the top_k / topk_group best experts (ties: lower index);
    5. renormalise the chosen scores to sum 1, times routed_scaling_factor.
    Slots are listed by descending key (ties: lower expert index).
    """
    if scoring == "softmax":
        raise ValueError("grouped top-k with softmax scoring: a softmax taken inside each group "
                         "sums to 1 in every group, so the group choice would rest on "
                         "tie-breaking alone")
    if scoring != "sigmoid":
        raise ValueError(f"unknown scoring function {scoring!r}")
    l32 = np.asarray(logits32, dtype=np.float32)
    T, E = l32.shape
    if n_group < 1 or E % n_group or not 1 <= topk_group <= n_group or top_k % topk_group:
        raise ValueError("grouped top-k needs E % n_group == 0, 1 <= topk_group <= n_group and "
                         "top_k % topk_group == 0")
    epg = E // n_group
    per = top_k // topk_group
    if per > epg:
        raise ValueError("top_k / topk_group exceeds the experts per group")
    s64 = sigmoid64(_selection_logits(l32).astype(np.float64))
    key = s64.astype(np.float32)
    groups = topk_desc(group_totals_fp32(key, n_group), topk_group)      # [T, topk_group]
    chosen = np.zeros((T, E), dtype=bool)
    rows = np.arange(T)[:, None]
    for r in range(topk_group):
        g = groups[:, r]
        cols = g[:, None] * epg + np.arange(epg)[None, :]
        inner = topk_desc(key[rows, cols], per)                            # [T, per]
        chosen[rows, np.take_along_axis(cols, inner, axis=1)] = True
    ids = topk_desc(np.where(chosen, key, np.float32(-np.inf)), top_k)
    ssel = np.take_along_axis(s64, ids, axis=1)
    w = ssel / np.sum(ssel, axis=1, keepdims=True) * routed_scaling_factor
    return ids.astype(np.int32), w


def route(logits, method: int, top_k: int, bias=None, n_group: int = 1, topk_group: int = 1,
          routed_scaling_factor: float = 1.0):
    """Routing: logits [T, E] fp32 -> (ids int32 [T, k], scales float64 [T, k]).

    TRT, section "路由方法枚举" (RoutingMethodType):
      Default (0)           softmax -> top-k, weights = selected softmax probabilities
      Renormalize (1)       top-k -> softmax over the selected logits
      DeepSeekV3 (2)        sigmoid -> bias add -> top-2 per group -> top groups -> top-k
      Llama4 (3)            top-k (Top1) -> sigmoid of each selected logit
      RenormalizeNaive (4)  softmax -> top-k -> divide by the selected sum
      MiniMax2 (5)          sigmoid -> bias add -> top-k -> divide by the unbiased sum
      SigmoidRenorm (6)     sigmoid -> top-k -> divide by the selected sum
    VLLM, section "FusedTopKRouter": the same softmax/sigmoid -> top-k -> renormalize.
    VLLM, section "GroupedTopKRouter": GROUPED_TOPK (16) = ``grouped_topk`` with sigmoid
    scoring; GROUPED_TOPK_SOFTMAX (17) is refused (see ``grouped_topk``).
    """
    l32 = np.asarray(logits, dtype=np.float32)
    T, E = l32.shape
    sel = _selection_logits(l32)
    l64 = sel.astype(np.float64)
    if method == LLAMA4:
        ids = topk_desc(sel, top_k)
        w = sigmoid64(np.take_along_axis(l64, ids, axis=1))
        return ids.astype(np.int32), w
    if method == MINIMAX2:
        b = np.zeros(E, np.float32) if bias is None else np.asarray(bias, np.float32)
        s64, kappa = deepseek_keys(l32, b)
        ids = topk_desc(kappa, top_k)
        ssel = np.take_along_axis(s64, ids, axis=1)
        w = ssel / np.sum(ssel, axis=1, keepdims=True)
        return ids.astype(np.int32), w
    if method in (DEFAULT, RENORMALIZE, RENORMALIZE_NAIVE, SIGMOID_RENORM):
        ids = topk_desc(sel, top_k)
        lsel = np.take_along_axis(l64, ids, axis=1)
        if method == DEFAULT:
            # The normaliser covers all E experts (TRT: Default vs Renormalize differ only
            # in which experts the denominator includes).
            w = np.take_along_axis(softmax64(l64), ids, axis=1)
        elif method == RENORMALIZE:
            w = softmax64(lsel)
        elif method == RENORMALIZE_NAIVE:
            p = np.take_along_axis(softmax64(l64), ids, axis=1)
            w = p / np.sum(p, axis=1, keepdims=True)
        else:
            s = sigmoid64(lsel)
            w = s / np.sum(s, axis=1, keepdims=True)
        return ids.astype(np.int32), w
    if method in (GROUPED_TOPK, GROUPED_TOPK_SOFTMAX):
        return grouped_topk(l32, top_k, n_group, topk_group, routed_scaling_factor,
                            "sigmoid" if method == GROUPED_TOPK else "softmax")
    if method == DEEPSEEKV3:
        b = np.zeros(E, np.float32) if bias is None else np.asarray(bias, np.float32)
        s64, kappa = deepseek_keys(l32, b)
        groups, _ = group_select(kappa, n_group, topk_group)
        epg = E // n_group
        in_group = np.zeros((T, n_group), dtype=bool)
        np.put_along_axis(in_group, groups, True, axis=1)
        mask = np.repeat(in_group, epg, axis=1)
        masked = np.where(mask, kappa, np.float32(-np.inf))
        ids = topk_desc(masked, top_k)
        ssel = np.take_along_axis(s64, ids, axis=1)
        w = ssel / (np.sum(ssel, axis=1, keepdims=True) + 1e-20) * routed_scaling_factor
        return ids.astype(np.int32), w
    raise ValueError(f"unsupported routing method {method}")


# --------------------------------------------------------------------------- permute

def permute(ids: np.ndarray, E: int):
    """Group the T*k (token, slot) pairs into contiguous per-expert blocks.

    GG section 2.1/2.2: all experts' rows are concatenated with an offset array;
    tokens are permuted so each expert's rows are contiguous. Within an expert the
    rows keep ascending flat index f = t*k + j (stable).
    Returns counts [E], offsets [E+1], perm_src [P] (position -> f), perm_inv [P].
    """
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    counts = np.bincount(flat, minlength=E)[:E]
    offsets = np.concatenate([[0], np.cumsum(counts)])
    perm_src = np.argsort(flat, kind="stable")
    perm_inv = np.empty_like(perm_src)
    perm_inv[perm_src] = np.arange(flat.size)
    return (counts.astype(np.int32), offsets.astype(np.int32), perm_src.astype(np.int32),
            perm_inv.astype(np.int32))


# --------------------------------------------------------------------------- experts

def swiglu(a: np.ndarray, I: int) -> np.ndarray:
    """h = silu(gate) * up with gate = a[:, :I], up = a[:, I:2I]."""
    g, u = a[:, :I], a[:, I:2 * I]
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g)) * u


def expert_ffn(X: np.ndarray, w13e, w2e) -> np.ndarray:
    """One SwiGLU expert on rows X [m, H]: w2e [H, I] . swiglu(w13e [2I, H] . x).

    VLLM, section "专家权重如何存储": w13 = gate and up merged, [2I, H]; w2 = down, [H, I].
    """
    w13e = np.asarray(w13e, dtype=np.float64)
    w2e = np.asarray(w2e, dtype=np.float64)
    I = w2e.shape[1]
    a = X @ w13e.T
    h = swiglu(a, I)
    return h @ w2e.T


def gate(x, wg, num_experts: int):
    """Router gate: logits = x . wg^T in float64. VLLM, section "Gate 计算与 FSE": with the
    fused shared-expert gate, wg has E + 1 rows and its last row gives the shared expert's
    gate logit. Returns (routed logits [T, E], shared logits [T] or None)."""
    X = np.asarray(x, dtype=np.float64)
    W = np.asarray(wg, dtype=np.float64)
    out = X @ W.T
    E = int(num_experts)
    return out[:, :E], (out[:, E] if W.shape[0] > E else None)


def _shared_weight(shared_gate, T):
    """Weight of the shared expert per token: 1, or sigmoid of its gate logit (VLLM, section
    "Gate 计算与 FSE": the shared expert's activation is usually a sigmoid)."""
    if shared_gate is None:
        return np.ones((T, 1))
    return sigmoid64(np.asarray(shared_gate, dtype=np.float64))[:, None]


def forward(x, ids, scales, w13, w2, w13_s=None, w2_s=None, shared_gate=None) -> np.ndarray:
    """y [T, H] float64 = sum_j scales[t, j] * E_{ids[t, j]}(x[t]) (+ g_t * shared(x[t]),
    g_t = 1 or sigmoid(shared_gate[t])).

    ``w13``/``w2`` are indexable per expert (``w13[e]`` -> [2I, H]), so callers can
    hand over one expert at a time. Tokens are independent: passing a subset of
    rows of x/ids/scales gives the matching rows of y.
    """
    X = np.asarray(x, dtype=np.float64)
    ids = np.asarray(ids)
    scales = np.asarray(scales, dtype=np.float64)
    T, H = X.shape
    y = np.zeros((T, H), dtype=np.float64)
    for e in np.unique(ids):
        rows, slots = np.nonzero(ids == e)
        o = expert_ffn(X[rows], w13[int(e)], w2[int(e)])
        np.add.at(y, rows, scales[rows, slots][:, None] * o)
    if w13_s is not None:
        y += _shared_weight(shared_gate, T) * expert_ffn(X, w13_s, w2_s)
    return y


def forward_partial(x, ids, scales, w13_local, w2_local, e_lo: int, e_hi: int, w13_s=None,
                    w2_s=None, shared_gate=None) -> np.ndarray:
    """The layer restricted to the experts [e_lo, e_hi): the slots whose expert lies
    there, weighted by their scales (+ the shared expert when given).

    TRT, section on supports_finalize_before_combine: with the top-k weighted sum taken
    on each rank's own rows, the slots of other ranks' experts contribute exactly 0, so
    the combine is an unweighted row sum. ``w13_local[e - e_lo]`` holds expert e.
    """
    X = np.asarray(x, dtype=np.float64)
    ids = np.asarray(ids)
    scales = np.asarray(scales, dtype=np.float64)
    T, H = X.shape
    y = np.zeros((T, H), dtype=np.float64)
    for e in range(e_lo, e_hi):
        rows, slots = np.nonzero(ids == e)
        if rows.size == 0:
            continue
        o = expert_ffn(X[rows], w13_local[e - e_lo], w2_local[e - e_lo])
        np.add.at(y, rows, scales[rows, slots][:, None] * o)
    if w13_s is not None:
        y += _shared_weight(shared_gate, T) * expert_ffn(X, w13_s, w2_s)
    return y


def forward_permuted(x, ids, scales, w13, w2, w13_s=None, w2_s=None):
    """The same result computed in the five-step order of the pages.

    route (given) -> permute -> per-expert FC1 + SwiGLU -> FC2 -> finalize (unpermute and
    apply the routing weights after FC2, TRT section on finalize before/after combine).
    Returns (y, intermediates) where intermediates holds counts/offsets/perm and the
    per-row h and FC2 outputs in permuted order (float64).
    """
    X = np.asarray(x, dtype=np.float64)
    ids = np.asarray(ids)
    T, k = ids.shape
    E = len(w13)
    counts, offsets, perm_src, perm_inv = permute(ids, E)
    x_perm = X[perm_src // k]
    I = np.asarray(w2[0]).shape[1]
    h = np.zeros((T * k, I))
    out = np.zeros((T * k, X.shape[1]))
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        if a == b:
            continue
        w13e = np.asarray(w13[e], dtype=np.float64)
        w2e = np.asarray(w2[e], dtype=np.float64)
        h[a:b] = swiglu(x_perm[a:b] @ w13e.T, I)
        out[a:b] = h[a:b] @ w2e.T
    sc = np.asarray(scales, dtype=np.float64).reshape(-1)
    y = np.zeros_like(X)
    for j in range(k):
        f = np.arange(T) * k + j
        y += sc[f][:, None] * out[perm_inv[f]]
    if w13_s is not None:
        y += expert_ffn(X, w13_s, w2_s)
    inter = dict(counts=counts, offsets=offsets, perm_src=perm_src, perm_inv=perm_inv,
                 h=h, out=out)
    return y, inter

"""The pins must catch plausible mistakes: each test plants one in the oracle (on the
CPU, through monkeypatch) and checks that a pin then fails."""
import numpy as np
import pytest

import oracle
import oracle.moe_oracle as om
import tests.test_oracle_pins as pins


def _fails(fn, *args):
    with pytest.raises(AssertionError):
        fn(*args)


def test_swapped_gate_up_is_caught(monkeypatch, golden_dir):
    def bad_swiglu(a, I):
        g, u = a[:, I:2 * I], a[:, :I]
        return g / (1.0 + np.exp(-g)) * u
    monkeypatch.setattr(om, "swiglu", bad_swiglu)
    _fails(pins.test_golden_ffn_and_layer, golden_dir)


def test_biased_weights_are_caught(monkeypatch, golden_dir):
    real = om.deepseek_keys

    def bad_keys(l, b):
        s64, kappa = real(l, b)
        return kappa.astype(np.float64), kappa   # weights would then use biased scores
    monkeypatch.setattr(om, "deepseek_keys", bad_keys)
    _fails(pins.test_golden_grouped_deepseek, golden_dir)


def test_full_group_sum_is_caught(monkeypatch, golden_dir):
    def bad_group_select(kappa, n_group, topk_group):
        T, E = kappa.shape
        gscore = kappa.reshape(T, n_group, E // n_group).sum(-1).astype(np.float32)
        return om.topk_desc(gscore, topk_group), gscore
    monkeypatch.setattr(om, "group_select", bad_group_select)
    _fails(pins.test_golden_grouped_deepseek, golden_dir)


def test_highest_index_tiebreak_is_caught(monkeypatch):
    def bad_topk(keys, k):
        rev = keys[..., ::-1]
        idx = np.argsort(-rev, axis=-1, kind="stable")[..., :k]
        return keys.shape[-1] - 1 - idx
    monkeypatch.setattr(om, "topk_desc", bad_topk)
    _fails(pins.test_topk_matches_rank_counting, oracle.RENORMALIZE)


def test_default_with_renorm_is_caught(monkeypatch):
    real = om.route

    def bad_route(logits, method, top_k, *a, **kw):
        if method == om.DEFAULT:
            method = om.RENORMALIZE_NAIVE
        return real(logits, method, top_k, *a, **kw)
    monkeypatch.setattr(om, "route", bad_route)
    monkeypatch.setattr(oracle, "route", bad_route)
    _fails(pins.test_weights_closed_forms)


def test_unstable_permute_is_caught(monkeypatch):
    def bad_permute(ids, E):
        flat = np.asarray(ids, dtype=np.int64).reshape(-1)
        counts = np.bincount(flat, minlength=E)[:E]
        offsets = np.concatenate([[0], np.cumsum(counts)])
        perm_src = np.lexsort((-np.arange(flat.size), flat))  # descending f inside a block
        perm_inv = np.empty_like(perm_src)
        perm_inv[perm_src] = np.arange(flat.size)
        return counts, offsets, perm_src, perm_inv
    monkeypatch.setattr(om, "permute", bad_permute)
    monkeypatch.setattr(oracle, "permute", bad_permute)
    _fails(pins.test_permute_brute_force_and_identity)


def test_renormalised_llama4_is_caught(monkeypatch, golden_dir):
    real = om.route

    def bad_route(logits, method, top_k, *a, **kw):
        if method == om.LLAMA4:
            method = om.SIGMOID_RENORM
        return real(logits, method, top_k, *a, **kw)
    monkeypatch.setattr(om, "route", bad_route)
    monkeypatch.setattr(oracle, "route", bad_route)
    _fails(pins.test_golden_llama4_and_minimax2, golden_dir)


def test_minimax2_biased_weights_are_caught(monkeypatch, golden_dir):
    real = om.deepseek_keys

    def bad_keys(l, b):
        s64, kappa = real(l, b)
        return kappa.astype(np.float64), kappa
    monkeypatch.setattr(om, "deepseek_keys", bad_keys)
    _fails(pins.test_golden_llama4_and_minimax2, golden_dir)


def test_minimax2_without_bias_is_caught(monkeypatch, golden_dir):
    real = om.deepseek_keys

    def bad_keys(l, b):
        return real(l, np.zeros_like(b))
    monkeypatch.setattr(om, "deepseek_keys", bad_keys)
    _fails(pins.test_golden_llama4_and_minimax2, golden_dir)


def test_partial_ignoring_scales_is_caught(monkeypatch):
    def bad_partial(x, ids, scales, w13_local, w2_local, e_lo, e_hi, w13_s=None, w2_s=None):
        X = np.asarray(x, dtype=np.float64)
        y = np.zeros_like(X)
        for e in range(e_lo, e_hi):
            rows, slots = np.nonzero(np.asarray(ids) == e)
            if rows.size:
                np.add.at(y, rows, om.expert_ffn(X[rows], w13_local[e - e_lo], w2_local[e - e_lo]))
        if w13_s is not None:
            y += om.expert_ffn(X, w13_s, w2_s)
        return y
    monkeypatch.setattr(om, "forward_partial", bad_partial)
    monkeypatch.setattr(oracle, "forward_partial", bad_partial)
    _fails(pins.test_partial_forward_partition_and_zeroed_scales)


def test_shared_gate_without_sigmoid_is_caught(monkeypatch):
    def bad_weight(shared_gate, T):
        if shared_gate is None:
            return np.ones((T, 1))
        return np.asarray(shared_gate, dtype=np.float64)[:, None]
    monkeypatch.setattr(om, "_shared_weight", bad_weight)
    _fails(pins.test_shared_gate_weight_limits_and_linearity)


def test_vllm_top2_group_score_is_caught(monkeypatch, golden_dir):
    def top2_totals(keys, n_group):
        T, E = keys.shape
        g = -np.sort(-keys.reshape(T, n_group, E // n_group), axis=-1)
        return (g[..., 0] + g[..., 1]).astype(np.float32)
    monkeypatch.setattr(om, "group_totals_fp32", top2_totals)
    _fails(pins.test_golden_vllm_grouped, golden_dir)


def test_vllm_global_topk_in_kept_groups_is_caught(monkeypatch, golden_dir):
    def global_topk(l32, top_k, n_group, topk_group, rsf=1.0, scoring="sigmoid"):
        T, E = l32.shape
        s64 = om.sigmoid64(l32.astype(np.float64))
        key = s64.astype(np.float32)
        groups = om.topk_desc(om.group_totals_fp32(key, n_group), topk_group)
        mask = np.zeros((T, n_group), bool)
        np.put_along_axis(mask, groups, True, axis=1)
        masked = np.where(np.repeat(mask, E // n_group, axis=1), key, np.float32(-np.inf))
        ids = om.topk_desc(masked, top_k)
        ssel = np.take_along_axis(s64, ids, axis=1)
        return ids.astype(np.int32), ssel / ssel.sum(1, keepdims=True) * rsf
    monkeypatch.setattr(om, "grouped_topk", global_topk)
    _fails(pins.test_golden_vllm_grouped, golden_dir)


def test_vllm_missing_renormalisation_is_caught(monkeypatch, golden_dir):
    real = om.grouped_topk

    def no_renorm(l32, top_k, n_group, topk_group, rsf=1.0, scoring="sigmoid"):
        ids, _ = real(l32, top_k, n_group, topk_group, rsf, scoring)
        s64 = om.sigmoid64(np.asarray(l32, np.float64))
        return ids, np.take_along_axis(s64, ids.astype(np.int64), axis=1) * rsf
    monkeypatch.setattr(om, "grouped_topk", no_renorm)
    _fails(pins.test_golden_vllm_grouped, golden_dir)

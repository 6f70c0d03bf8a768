"""Pins for the CPU oracle: hand-worked examples, brute force, closed forms, invariants.

Each check is independent of the oracle's own code path (rank counting instead of
sorting, subset enumeration instead of top-k, explicit Python loops instead of
matrix products, closed-form values from the golden fixtures).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import (DEFAULT, RENORMALIZE, DEEPSEEKV3, LLAMA4, RENORMALIZE_NAIVE, MINIMAX2,
                    SIGMOID_RENORM, GROUPED_TOPK, GROUPED_TOPK_SOFTMAX)


def _ev(expr):
    return float(eval(expr, {"__builtins__": {}}, {"exp": math.exp, "log": math.log}))


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- golden fixtures

def test_golden_softmax_family(golden_dir):
    g = _load(golden_dir, "route_softmax_hand.json")
    for case in g["cases"]:
        logits = np.array([[_ev(e) for e in case["logits_expr"]]], np.float32)
        for m_str, exprs in case["scales_expr"].items():
            ids, sc = oracle.route(logits, int(m_str), case["top_k"])
            assert ids[0].tolist() == case["expected_ids"], (m_str, ids)
            np.testing.assert_allclose(sc[0], [_ev(e) for e in exprs], rtol=1e-6)


def test_golden_grouped_deepseek(golden_dir):
    g = _load(golden_dir, "route_grouped_hand.json")
    p = np.array(g["probabilities"], np.float64)
    logits = np.log(p / (1 - p)).astype(np.float32)[None, :]
    bias = np.array(g["bias"], np.float32)
    s64, kappa = oracle.deepseek_keys(logits, bias)
    groups, _ = oracle.group_select(kappa, g["n_group"], g["topk_group"])
    assert groups[0].tolist() == g["expected_groups"]
    ids, sc = oracle.route(logits, DEEPSEEKV3, g["top_k"], bias=bias, n_group=g["n_group"],
                           topk_group=g["topk_group"],
                           routed_scaling_factor=g["routed_scaling_factor"])
    assert ids[0].tolist() == g["expected_ids"]
    np.testing.assert_allclose(sc[0], [_ev(e) for e in g["expected_scales_expr"]], rtol=1e-6)


def test_golden_vllm_grouped(golden_dir):
    g = _load(golden_dir, "route_vllm_grouped_hand.json")
    p = np.array(g["probabilities"], np.float64)
    logits = np.log(p / (1 - p)).astype(np.float32)[None, :]
    key = oracle.sigmoid64(logits.astype(np.float64)).astype(np.float32)
    epg = g["E"] // g["n_group"]
    sums = [sum(g["probabilities"][j * epg:(j + 1) * epg]) for j in range(g["n_group"])]
    np.testing.assert_allclose(oracle.group_totals_fp32(key, g["n_group"])[0], sums, rtol=1e-6)
    ids, sc = oracle.route(logits, GROUPED_TOPK, g["top_k"], n_group=g["n_group"],
                           topk_group=g["topk_group"],
                           routed_scaling_factor=g["routed_scaling_factor"])
    assert ids[0].tolist() == g["expected_ids"]
    assert sorted({e // epg for e in ids[0].tolist()}) == sorted(g["expected_groups"])
    np.testing.assert_allclose(sc[0], [_ev(e) for e in g["expected_scales_expr"]], rtol=1e-6)


def test_golden_llama4_and_minimax2(golden_dir):
    g = _load(golden_dir, "route_llama4_minimax_hand.json")
    for case in g["llama4"]:
        logits = np.array([[_ev(e) for e in case["logits_expr"]]], np.float32)
        ids, sc = oracle.route(logits, LLAMA4, case["top_k"])
        assert ids[0].tolist() == case["expected_ids"]
        np.testing.assert_allclose(sc[0], [_ev(e) for e in case["scales_expr"]], rtol=1e-6)
    for case in g["minimax2"]:
        p = np.array(case["probabilities"], np.float64)
        logits = np.log(p / (1 - p)).astype(np.float32)[None, :]
        ids, sc = oracle.route(logits, MINIMAX2, case["top_k"],
                               bias=np.array(case["bias"], np.float32))
        assert ids[0].tolist() == case["expected_ids"]
        np.testing.assert_allclose(sc[0], [_ev(e) for e in case["scales_expr"]], rtol=1e-6)


def test_golden_ffn_and_layer(golden_dir):
    g = _load(golden_dir, "ffn_hand.json")
    w13 = np.array(g["w13"], np.float64)
    w2 = np.array(g["w2"], np.float64)
    x = np.array(g["x"], np.float64)
    for e_str, rows in g["expert_outputs_expr"].items():
        got = oracle.expert_ffn(x, w13[int(e_str)], w2[int(e_str)])
        want = np.array([[_ev(v) for v in r] for r in rows])
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-15)
    lay = g["layer"]
    want = np.array([[_ev(v) for v in r] for r in lay["expected_expr"]])
    ids = np.array(lay["ids"])
    sc = np.array(lay["scales"])
    np.testing.assert_allclose(oracle.forward(x, ids, sc, w13, w2), want, rtol=1e-12)
    y2, _ = oracle.forward_permuted(x, ids, sc, w13, w2)
    np.testing.assert_allclose(y2, want, rtol=1e-12)


def test_golden_permute(golden_dir):
    g = _load(golden_dir, "permute_hand.json")
    counts, offsets, perm_src, perm_inv = oracle.permute(np.array(g["ids"]), g["E"])
    assert counts.tolist() == g["expected_counts"]
    assert offsets.tolist() == g["expected_offsets"]
    assert perm_src.tolist() == g["expected_perm_src"]
    assert perm_inv.tolist() == g["expected_perm_inv"]


# ---------------------------------------------------------------- brute force: top-k

def _rank_select(keys, k):
    """Expert e is chosen iff fewer than k experts beat it; beat = larger key, or the
    same key and a lower index. Its slot is that count. No sorting involved."""
    E = len(keys)
    out = [None] * k
    for e in range(E):
        beat = sum(1 for o in range(E) if keys[o] > keys[e] or (keys[o] == keys[e] and o < e))
        if beat < k:
            out[beat] = e
    return out


@pytest.mark.parametrize("method", [DEFAULT, RENORMALIZE, LLAMA4, RENORMALIZE_NAIVE,
                                    SIGMOID_RENORM])
def test_topk_matches_rank_counting(method):
    rng = np.random.default_rng(1)
    for trial in range(60):
        E = int(rng.integers(1, 13))
        k = int(rng.integers(1, E + 1))
        T = 5
        if trial % 3 == 0:  # many exact ties
            logits = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
        else:
            logits = rng.standard_normal((T, E)).astype(np.float32)
        ids, sc = oracle.route(logits, method, k)
        for t in range(T):
            assert ids[t].tolist() == _rank_select(logits[t].tolist(), k)
            assert len(set(ids[t].tolist())) == k


def _softmax_loop(v):
    m = max(v)
    z = [math.exp(a - m) for a in v]
    s = sum(z)
    return [a / s for a in z]


def test_weights_closed_forms():
    rng = np.random.default_rng(2)
    T, E, k = 16, 10, 4
    logits = rng.standard_normal((T, E)).astype(np.float32)
    for t in range(T):
        l = [float(a) for a in logits[t]]
        sel = _rank_select(l, k)
        p = _softmax_loop(l)
        sig = [1 / (1 + math.exp(-l[e])) for e in sel]
        want = {
            DEFAULT: [p[e] for e in sel],
            RENORMALIZE: _softmax_loop([l[e] for e in sel]),
            RENORMALIZE_NAIVE: [p[e] / sum(p[s] for s in sel) for e in sel],
            SIGMOID_RENORM: [s / sum(sig) for s in sig],
            LLAMA4: sig,
        }
        for m, w in want.items():
            _, sc = oracle.route(logits[t:t + 1], m, k)
            np.testing.assert_allclose(sc[0], w, rtol=1e-12)


def test_renormalize_equals_naive_and_sums():
    rng = np.random.default_rng(3)
    logits = (3 * rng.standard_normal((200, 64))).astype(np.float32)
    i1, s1 = oracle.route(logits, RENORMALIZE, 6)
    i4, s4 = oracle.route(logits, RENORMALIZE_NAIVE, 6)
    i6, s6 = oracle.route(logits, SIGMOID_RENORM, 6)
    i0, s0 = oracle.route(logits, DEFAULT, 6)
    assert (i1 == i4).all() and (i1 == i6).all() and (i1 == i0).all()
    np.testing.assert_allclose(s1, s4, rtol=1e-12)
    np.testing.assert_allclose(s1.sum(1), 1, rtol=1e-12)
    np.testing.assert_allclose(s6.sum(1), 1, rtol=1e-12)
    assert (s0.sum(1) <= 1 + 1e-12).all()
    # Default weights are the selected softmax probabilities: descending like the logits
    assert (np.diff(s0, axis=1) <= 0).all()


# ---------------------------------------------------------------- brute force: groups

def _grouped_brute(logit, bias, n_group, topk_group, k, rsf):
    """Enumerate every topk_group-subset of groups; keep the one with the largest sum
    of group scores (then the lexicographically smallest sorted index tuple); choose
    experts by rank counting inside the union."""
    E = len(logit)
    epg = E // n_group
    s = [1 / (1 + math.exp(-float(v))) for v in logit]
    kappa = [float(np.float32(np.float32(si) + np.float32(b))) for si, b in zip(s, bias)]
    gs = []
    for g in range(n_group):
        vals = sorted(kappa[g * epg:(g + 1) * epg], reverse=True)
        gs.append(float(np.float32(np.float32(vals[0]) + np.float32(vals[1]))))
    best = None
    for sub in itertools.combinations(range(n_group), topk_group):
        tot = sum(gs[g] for g in sub)
        if best is None or tot > best[0]:
            best = (tot, sub)
    chosen = set(best[1])
    keys = [kappa[e] if e // epg in chosen else -math.inf for e in range(E)]
    sel = _rank_select(keys, k)
    ssel = [s[e] for e in sel]
    w = [v / (sum(ssel) + 1e-20) * rsf for v in ssel]
    return chosen, sel, w, gs


def test_grouped_routing_matches_subset_enumeration():
    rng = np.random.default_rng(4)
    for trial in range(150):
        n_group = int(rng.integers(2, 6))
        epg = int(rng.integers(2, 6))
        E = n_group * epg
        topk_group = int(rng.integers(1, n_group + 1))
        k = int(rng.integers(1, topk_group * epg + 1))
        logits = rng.standard_normal((1, E)).astype(np.float32)
        bias = (0.1 * rng.standard_normal(E)).astype(np.float32)
        rsf = float(rng.choice([1.0, 2.5]))
        chosen, sel, w, gs = _grouped_brute(logits[0], bias, n_group, topk_group, k, rsf)
        sorted_gs = sorted(gs, reverse=True)
        if topk_group < n_group and sorted_gs[topk_group - 1] == sorted_gs[topk_group]:
            continue  # tied boundary: subset choice not unique by the sum criterion
        ids, sc = oracle.route(logits, DEEPSEEKV3, k, bias=bias, n_group=n_group,
                               topk_group=topk_group, routed_scaling_factor=rsf)
        assert ids[0].tolist() == sel
        assert all(e // epg in chosen for e in ids[0])
        np.testing.assert_allclose(sc[0], w, rtol=1e-12)
        np.testing.assert_allclose(sc[0].sum(), rsf * sum(1 / (1 + math.exp(-float(logits[0, e])))
                                   for e in sel) / (sum(1 / (1 + math.exp(-float(logits[0, e])))
                                                        for e in sel) + 1e-20), rtol=1e-12)


def test_grouped_single_group_reduces_to_sigmoid_renorm():
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((64, 32)).astype(np.float32)
    ia, sa = oracle.route(logits, DEEPSEEKV3, 4, bias=np.zeros(32, np.float32), n_group=1,
                          topk_group=1, routed_scaling_factor=1.0)
    ib, sb = oracle.route(logits, SIGMOID_RENORM, 4)
    # distinct logits can share one fp32 sigmoid value; compare the chosen key values
    s = oracle.sigmoid64(logits.astype(np.float64)).astype(np.float32)
    assert (np.take_along_axis(s, ia, 1) == np.take_along_axis(s, ib, 1)).all()
    same = (ia == ib).all(1)
    assert same.mean() > 0.9
    np.testing.assert_allclose(sa[same], sb[same], rtol=1e-12)


def _vllm_grouped_brute(logit, n_group, topk_group, k, rsf):
    """vLLM grouped top-k by enumeration: the group totals added one fp32 step at a time in
    expert order; the topk_group-subset of groups with the largest sum of totals (then the
    lexicographically smallest index tuple, i.e. lower group indices win ties); inside each
    kept group its k / topk_group experts by rank counting; slots by rank counting over the
    union; weights from explicit loops over the float64 sigmoid."""
    E = len(logit)
    epg = E // n_group
    per = k // topk_group
    s = [1 / (1 + math.exp(-float(v))) for v in logit]
    key = [float(np.float32(si)) for si in s]
    totals = []
    for g in range(n_group):
        acc = np.float32(key[g * epg])
        for j in range(1, epg):
            acc = np.float32(acc + np.float32(key[g * epg + j]))
        totals.append(float(acc))
    best = None
    for sub in itertools.combinations(range(n_group), topk_group):
        tot = sum(totals[g] for g in sub)
        if best is None or tot > best[0]:
            best = (tot, sub)
    chosen = []
    for g in best[1]:
        chosen += [g * epg + e for e in _rank_select(key[g * epg:(g + 1) * epg], per)]
    order = _rank_select([key[e] if e in chosen else -math.inf for e in range(E)], k)
    ssel = [s[e] for e in order]
    return set(best[1]), order, [v / sum(ssel) * rsf for v in ssel]


def test_vllm_grouped_matches_subset_enumeration():
    rng = np.random.default_rng(12)
    for trial in range(200):
        n_group = int(rng.integers(1, 6))
        epg = int(rng.integers(1, 7))
        E = n_group * epg
        topk_group = int(rng.integers(1, n_group + 1))
        per = int(rng.integers(1, epg + 1))
        k = per * topk_group
        if trial % 3 == 0:   # exact ties in keys and group totals
            logits = rng.integers(-2, 3, size=(1, E)).astype(np.float32)
        else:
            logits = rng.standard_normal((1, E)).astype(np.float32)
        rsf = float(rng.choice([1.0, 2.5]))
        chosen, sel, w = _vllm_grouped_brute(logits[0], n_group, topk_group, k, rsf)
        ids, sc = oracle.route(logits, GROUPED_TOPK, k, n_group=n_group, topk_group=topk_group,
                               routed_scaling_factor=rsf)
        assert ids[0].tolist() == sel, (trial, ids, sel)
        assert {e // epg for e in ids[0].tolist()} == chosen
        for g in chosen:   # exactly k / topk_group experts from every kept group
            assert sum(1 for e in ids[0].tolist() if e // epg == g) == per
        np.testing.assert_allclose(sc[0], w, rtol=1e-12)
        np.testing.assert_allclose(sc[0].sum(), rsf, rtol=1e-12)


def test_vllm_grouped_reductions():
    rng = np.random.default_rng(13)
    logits = rng.standard_normal((64, 32)).astype(np.float32)
    # one group: the per-group top-k is the plain top-k of the sigmoid scores
    ia, sa = oracle.route(logits, GROUPED_TOPK, 4, n_group=1, topk_group=1)
    ib, sb = oracle.route(logits, SIGMOID_RENORM, 4)
    s = oracle.sigmoid64(logits.astype(np.float64)).astype(np.float32)
    assert (np.take_along_axis(s, ia, 1) == np.take_along_axis(s, ib, 1)).all()
    same = (ia == ib).all(1)
    assert same.mean() > 0.9
    np.testing.assert_allclose(sa[same], sb[same], rtol=1e-12)
    # every expert of a kept group chosen: the kept groups are the top groups by total
    ids, _ = oracle.route(logits, GROUPED_TOPK, 8, n_group=8, topk_group=2)
    for t in range(64):
        tot = [sum(float(v) for v in s[t, g * 4:(g + 1) * 4]) for g in range(8)]
        top = sorted(range(8), key=lambda g: (-tot[g], g))[:2]
        assert sorted(ids[t].tolist()) == sorted(e for g in top for e in range(4 * g, 4 * g + 4))
    # softmax scoring is refused: its group totals are 1 in every group
    with pytest.raises(ValueError, match="sums to 1"):
        oracle.route(logits, GROUPED_TOPK_SOFTMAX, 4, n_group=8, topk_group=2)
    with pytest.raises(ValueError):
        oracle.route(logits, GROUPED_TOPK, 5, n_group=8, topk_group=2)   # 5 % 2 != 0


def test_bias_moves_selection_not_weights():
    rng = np.random.default_rng(6)
    T, E = 64, 32
    logits = rng.standard_normal((T, E)).astype(np.float32)
    b = (0.5 * rng.standard_normal(E)).astype(np.float32)
    ib, sb = oracle.route(logits, DEEPSEEKV3, 4, bias=b, n_group=4, topk_group=2)
    i0, s0 = oracle.route(logits, DEEPSEEKV3, 4, bias=np.zeros(E, np.float32), n_group=4,
                          topk_group=2)
    assert (ib != i0).any()  # the bias does change who is chosen
    sig = oracle.sigmoid64(logits.astype(np.float64))
    for t in range(T):
        v = sig[t, ib[t]]
        np.testing.assert_allclose(sb[t], v / (v.sum() + 1e-20), rtol=1e-12)


def test_minimax2_brute_force_and_single_group_deepseek():
    rng = np.random.default_rng(7)
    for trial in range(30):
        E = int(rng.integers(2, 40))
        k = int(rng.integers(1, min(E, 8) + 1))
        T = 6
        if trial % 3 == 0:   # exact ties in the keys
            logits = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
            b = np.zeros(E, np.float32)
        else:
            logits = rng.standard_normal((T, E)).astype(np.float32)
            b = (0.3 * rng.standard_normal(E)).astype(np.float32)
        ids, sc = oracle.route(logits, MINIMAX2, k, bias=b)
        for t in range(T):
            # keys by rank counting; weights by explicit loops over the unbiased sigmoid
            kappa = [float(np.float32(np.float32(1 / (1 + math.exp(-float(l)))) + bb))
                     for l, bb in zip(logits[t], b)]
            sel = _rank_select(kappa, k)
            assert ids[t].tolist() == sel
            sig = [1 / (1 + math.exp(-float(logits[t][e]))) for e in sel]
            np.testing.assert_allclose(sc[t], [v / sum(sig) for v in sig], rtol=1e-12)
        i2, s2 = oracle.route(logits, DEEPSEEKV3, k, bias=b, n_group=1, topk_group=1,
                              routed_scaling_factor=1.0)
        assert np.array_equal(ids, i2)
        np.testing.assert_allclose(sc, s2, rtol=1e-12)


# ---------------------------------------------------------------- permute

def test_permute_brute_force_and_identity():
    rng = np.random.default_rng(7)
    for trial in range(20):
        E = int(rng.integers(1, 20))
        T = int(rng.integers(0, 50))
        k = int(rng.integers(1, min(E, 4) + 1))
        ids = rng.integers(0, E, size=(T, k))
        counts, offsets, perm_src, perm_inv = oracle.permute(ids, E)
        flat = ids.reshape(-1).tolist()
        order = sorted(range(len(flat)), key=lambda f: (flat[f], f))
        assert perm_src.tolist() == order
        assert counts.tolist() == [flat.count(e) for e in range(E)]
        assert offsets[0] == 0 and offsets[-1] == T * k and (np.diff(offsets) >= 0).all()
        assert (perm_inv[perm_src] == np.arange(T * k)).all()
        assert (perm_src[perm_inv] == np.arange(T * k)).all()
        # every row sits inside its expert's block
        for f, e in enumerate(flat):
            assert offsets[e] <= perm_inv[f] < offsets[e + 1]
        # permute then unpermute is the identity on row payloads
        payload = rng.standard_normal((T * k, 3))
        assert np.array_equal(payload[perm_src][perm_inv], payload)


# ---------------------------------------------------------------- experts / layer

def _dense_ffn_loops(x, w13, w2):
    """y = W2 . (silu(W1 x) * (W3 x)) with explicit loops (tiny sizes only)."""
    H = len(x)
    I = len(w2[0])
    h = []
    for i in range(I):
        g = sum(w13[i][c] * x[c] for c in range(H))
        u = sum(w13[I + i][c] * x[c] for c in range(H))
        h.append(g / (1 + math.exp(-g)) * u)
    return [sum(w2[r][i] * h[i] for i in range(I)) for r in range(H)]


def test_single_expert_top1_is_dense_ffn():
    rng = np.random.default_rng(8)
    T, H, I = 5, 6, 4
    x = rng.standard_normal((T, H))
    w13 = rng.standard_normal((1, 2 * I, H))
    w2 = rng.standard_normal((1, H, I))
    logits = rng.standard_normal((T, 1)).astype(np.float32)
    for m in (RENORMALIZE, RENORMALIZE_NAIVE, SIGMOID_RENORM, DEFAULT):
        ids, sc = oracle.route(logits, m, 1)
        assert (ids == 0).all()
        np.testing.assert_allclose(sc, 1.0, rtol=1e-15)
        y = oracle.forward(x, ids, sc, w13, w2)
        for t in range(T):
            np.testing.assert_allclose(y[t], _dense_ffn_loops(x[t].tolist(), w13[0].tolist(),
                                                               w2[0].tolist()), rtol=1e-10)


def test_layer_against_loops_linearity_and_equivariance():
    rng = np.random.default_rng(9)
    T, H, I, E, k = 7, 5, 3, 4, 2
    x = rng.standard_normal((T, H))
    w13 = rng.standard_normal((E, 2 * I, H))
    w2 = rng.standard_normal((E, H, I))
    w13s = rng.standard_normal((2 * I, H))
    w2s = rng.standard_normal((H, I))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    sc = rng.random((T, k))
    y = oracle.forward(x, ids, sc, w13, w2, w13s, w2s)
    for t in range(T):
        want = np.array(_dense_ffn_loops(x[t].tolist(), w13s.tolist(), w2s.tolist()))
        for j in range(k):
            want += sc[t, j] * np.array(_dense_ffn_loops(x[t].tolist(), w13[ids[t, j]].tolist(),
                                                         w2[ids[t, j]].tolist()))
        np.testing.assert_allclose(y[t], want, rtol=1e-10)
    # the five-step order gives the same result
    y5, inter = oracle.forward_permuted(x, ids, sc, w13, w2, w13s, w2s)
    np.testing.assert_allclose(y5, y, rtol=1e-12)
    # linear in the routing scales (shared part fixed)
    ys = oracle.forward(x, ids, np.zeros_like(sc), w13, w2, w13s, w2s)
    y2 = oracle.forward(x, ids, 2 * sc, w13, w2, w13s, w2s)
    np.testing.assert_allclose(y2 - ys, 2 * (y - ys), rtol=1e-10, atol=1e-12)
    # zero routed scales leave the shared expert alone = dense FFN
    for t in range(T):
        np.testing.assert_allclose(ys[t], _dense_ffn_loops(x[t].tolist(), w13s.tolist(),
                                                           w2s.tolist()), rtol=1e-10)
    # permuting tokens permutes rows of y
    pi = rng.permutation(T)
    yp = oracle.forward(x[pi], ids[pi], sc[pi], w13, w2, w13s, w2s)
    np.testing.assert_allclose(yp, y[pi], rtol=1e-12)
    # duplicate ids are independent rows
    ids_dup = ids.copy()
    ids_dup[:, 1] = ids_dup[:, 0]
    yd = oracle.forward(x, ids_dup, sc, w13, w2)
    for t in range(T):
        e = ids_dup[t, 0]
        want = (sc[t, 0] + sc[t, 1]) * np.array(_dense_ffn_loops(x[t].tolist(), w13[e].tolist(),
                                                                 w2[e].tolist()))
        np.testing.assert_allclose(yd[t], want, rtol=1e-10)


def test_partial_forward_partition_and_zeroed_scales():
    """The expert-range forward: partials over a partition of [0, E) (the shared expert in
    one of them) add up to the layer; each partial equals the layer with the scales of
    the other experts' slots set to 0 (a different computation: all experts run)."""
    rng = np.random.default_rng(9)
    T, H, I, E, k, Is = 12, 6, 5, 6, 3, 4
    x = rng.standard_normal((T, H))
    w13 = rng.standard_normal((E, 2 * I, H)) * 0.5
    w2 = rng.standard_normal((E, H, I)) * 0.5
    w13s = rng.standard_normal((2 * Is, H)) * 0.5
    w2s = rng.standard_normal((H, Is)) * 0.5
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    scales = rng.random((T, k))
    full = oracle.forward(x, ids, scales, w13, w2, w13s, w2s)
    cuts = [(0, 2), (2, 5), (5, 6)]
    parts = []
    for n, (lo, hi) in enumerate(cuts):
        sh = (w13s, w2s) if n == 0 else (None, None)
        parts.append(oracle.forward_partial(x, ids, scales, w13[lo:hi], w2[lo:hi], lo, hi, *sh))
        zeroed = np.where((ids >= lo) & (ids < hi), scales, 0.0)
        np.testing.assert_allclose(parts[-1], oracle.forward(x, ids, zeroed, w13, w2, *sh),
                                   rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sum(parts), full, rtol=1e-12, atol=1e-12)


def test_gate_is_the_plain_product_and_splits_the_shared_row():
    rng = np.random.default_rng(10)
    T, H, E = 5, 7, 4
    x = rng.standard_normal((T, H))
    wg = rng.standard_normal((E + 1, H))
    routed, shared = oracle.gate(x, wg, E)
    for t in range(T):
        for e in range(E + 1):
            want = sum(x[t, h] * wg[e, h] for h in range(H))
            got = routed[t, e] if e < E else shared[t]
            assert abs(got - want) <= 1e-12 * max(1.0, abs(want))
    r2, s2 = oracle.gate(x, wg[:E], E)
    assert s2 is None and np.array_equal(r2, routed)


def test_shared_gate_weight_limits_and_linearity():
    """The fused shared-expert gate scales the shared expert by sigmoid(g): g -> +inf gives
    the ungated layer, g -> -inf the routed part alone, and in between the layer is
    routed + sigmoid(g) * (ungated - routed)."""
    rng = np.random.default_rng(11)
    T, H, I, E, k, Is = 6, 5, 4, 3, 2, 3
    x = rng.standard_normal((T, H))
    w13 = rng.standard_normal((E, 2 * I, H))
    w2 = rng.standard_normal((E, H, I))
    w13s = rng.standard_normal((2 * Is, H))
    w2s = rng.standard_normal((H, Is))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    sc = rng.random((T, k))
    ungated = oracle.forward(x, ids, sc, w13, w2, w13s, w2s)
    routed = oracle.forward(x, ids, sc, w13, w2)
    np.testing.assert_allclose(oracle.forward(x, ids, sc, w13, w2, w13s, w2s,
                                              shared_gate=np.full(T, 60.0)), ungated, rtol=1e-12)
    np.testing.assert_allclose(oracle.forward(x, ids, sc, w13, w2, w13s, w2s,
                                              shared_gate=np.full(T, -60.0)), routed,
                               rtol=1e-12, atol=1e-20)
    g = rng.standard_normal(T)
    sig = np.array([1 / (1 + math.exp(-v)) for v in g])[:, None]
    np.testing.assert_allclose(oracle.forward(x, ids, sc, w13, w2, w13s, w2s, shared_gate=g),
                               routed + sig * (ungated - routed), rtol=1e-12, atol=1e-12)


def test_empty_and_degenerate():
    ids, sc = oracle.route(np.zeros((0, 8), np.float32), RENORMALIZE_NAIVE, 2)
    assert ids.shape == (0, 2) and sc.shape == (0, 2)
    c, o, ps, pi = oracle.permute(np.zeros((0, 2), np.int32), 8)
    assert c.sum() == 0 and o.tolist() == [0] * 9 and ps.size == 0
    y = oracle.forward(np.zeros((0, 4)), np.zeros((0, 2), np.int32), np.zeros((0, 2)),
                       np.zeros((8, 6, 4)), np.zeros((8, 4, 3)))
    assert y.shape == (0, 4)
    # k = E: every expert selected, listed by descending logit
    logits = np.array([[0.5, -1.0, 2.0, 0.0]], np.float32)
    ids, sc = oracle.route(logits, RENORMALIZE, 4)
    assert ids[0].tolist() == [2, 0, 3, 1]
    np.testing.assert_allclose(sc[0], oracle.softmax64(logits.astype(np.float64))[0][[2, 0, 3, 1]],
                               rtol=1e-12)
    # non-finite logits are never preferred over finite ones
    logits = np.array([[np.nan, 1.0, np.inf, 0.0]], np.float32)
    ids, _ = oracle.route(logits, RENORMALIZE_NAIVE, 2)
    assert ids[0].tolist() == [1, 3]

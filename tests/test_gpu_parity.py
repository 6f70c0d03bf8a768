"""GPU parity: the CUDA path (called through the C ABI) against the CPU oracle on the same
seeded inputs. Expert ids, counts, offsets and the permutation must match bit for bit;
routing scales within 1e-6 relative; h / FC2 rows / y within max|err| <= tol * max|ref|
(y: 2e-2, the bf16 output tolerance; the oracle accumulates in fp64)."""
import numpy as np
import pytest
import torch

import oracle
from workloads import (WORKLOADS, Workload, make_inputs, DEFAULT, RENORMALIZE, DEEPSEEKV3,
                       LLAMA4, RENORMALIZE_NAIVE, MINIMAX2, SIGMOID_RENORM, GROUPED_TOPK)

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

Y_TOL = 2e-2
H_TOL = 1e-2


@pytest.fixture(scope="module")
def moe():
    import mixture_experts_layer_03_gb300 as m
    return m


class ExpertView:
    """Per-expert host float64 copies of a device weight tensor (one expert at a time)."""

    def __init__(self, t):
        self.t = t

    def __len__(self):
        return self.t.shape[0]

    def __getitem__(self, e):
        return self.t[int(e)].cpu().double().numpy()


def _np64(t):
    return t.cpu().double().numpy()


def _check_close(got, ref, tol, what):
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref).max() if ref.size else 0.0
    bound = tol * (np.abs(ref).max() if ref.size else 0.0)
    assert err <= bound, f"{what}: max|err| = {err:.4e} > {bound:.4e}"
    return err, bound


def _to_bf16_dev(moe, t, dev="cuda"):
    t = t.to(dev)
    return moe.moe_cast_f32_to_bf16(t) if t.dtype == torch.float32 else t


# ------------------------------------------------------------------------ routing

ROUTE_CASES = [
    # (T, E, k, method, n_group, topk_group, rsf, logit_scale, int_logits)
    (257, 8, 2, RENORMALIZE_NAIVE, 1, 1, 1.0, 1.0, False),
    (100, 8, 2, DEFAULT, 1, 1, 1.0, 1.0, False),
    (100, 64, 6, RENORMALIZE, 1, 1, 1.0, 3.0, False),
    (100, 128, 8, SIGMOID_RENORM, 1, 1, 1.0, 1.0, False),
    (100, 256, 8, DEEPSEEKV3, 8, 4, 2.5, 1.0, False),
    (100, 96, 5, DEEPSEEKV3, 4, 2, 1.0, 1.0, False),
    (100, 33, 3, RENORMALIZE_NAIVE, 1, 1, 1.0, 1.0, False),   # E not a multiple of 32
    (64, 16, 4, RENORMALIZE_NAIVE, 1, 1, 1.0, 1.0, True),     # many exact ties
    (64, 16, 4, DEEPSEEKV3, 4, 2, 1.0, 1.0, True),            # ties in keys and group scores
    (64, 1, 1, SIGMOID_RENORM, 1, 1, 1.0, 1.0, False),        # one expert
    (64, 8, 8, DEFAULT, 1, 1, 1.0, 1.0, False),               # k = E
    (1, 256, 8, RENORMALIZE, 1, 1, 1.0, 1.0, False),          # one token
    (257, 16, 1, LLAMA4, 1, 1, 1.0, 1.0, False),              # Top1 -> sigmoid
    (100, 128, 1, LLAMA4, 1, 1, 1.0, 3.0, False),
    (64, 16, 4, LLAMA4, 1, 1, 1.0, 1.0, True),                # k > 1, exact ties
    (257, 256, 8, MINIMAX2, 1, 1, 1.0, 1.0, False),           # biased keys over all 256
    (100, 64, 4, MINIMAX2, 1, 1, 1.0, 1.0, False),
    (64, 16, 4, MINIMAX2, 1, 1, 1.0, 1.0, True),              # ties in the keys
    (257, 256, 8, GROUPED_TOPK, 8, 4, 2.5, 1.0, False),       # vLLM grouped: 2 from 4 of 8 groups
    (100, 64, 6, GROUPED_TOPK, 8, 3, 1.0, 1.0, False),
    (64, 16, 4, GROUPED_TOPK, 4, 2, 1.0, 1.0, True),          # ties in keys and group totals
    (100, 96, 4, GROUPED_TOPK, 1, 1, 1.0, 1.0, False),        # one group of 96
    (100, 32, 8, GROUPED_TOPK, 32, 8, 1.0, 1.0, False),       # one expert per group
    (100, 128, 8, GROUPED_TOPK, 16, 2, 1.0, 3.0, False),      # 4 from 2 of 16 groups
]


def _random_route_cases(n, seed):
    """Seeded random routing problems inside the envelope, every method, with random valid
    group parameters for the grouped ones; half of them draw integer logits (exact ties in
    logits, keys and group scores)."""
    rng = np.random.default_rng(seed)
    methods = [DEFAULT, RENORMALIZE, DEEPSEEKV3, LLAMA4, RENORMALIZE_NAIVE, MINIMAX2,
               SIGMOID_RENORM, GROUPED_TOPK]
    cases = []
    for i in range(n):
        method = methods[i % len(methods)]
        T = int(rng.integers(1, 600))
        ng, tg, rsf = 1, 1, 1.0
        if method == DEEPSEEKV3:
            ng = int(rng.choice([1, 2, 4, 8, 16]))
            epg = int(rng.integers(2, min(32, 256 // ng) + 1))
            E = ng * epg
            tg = int(rng.integers(1, ng + 1))
            while epg * tg > 256:
                tg -= 1
            k = int(rng.integers(1, min(8, epg * tg) + 1))
            rsf = float(rng.choice([1.0, 2.5]))
        elif method == GROUPED_TOPK:
            ng = int(rng.choice([1, 2, 4, 8, 16, 32]))
            epg = int(rng.integers(1, max(1, 256 // ng) + 1))
            E = ng * epg
            tg = int(rng.integers(1, min(ng, 8) + 1))
            per = int(rng.integers(1, min(epg, 8 // tg) + 1))
            k = per * tg
            rsf = float(rng.choice([1.0, 2.5]))
        else:
            E = int(rng.integers(1, 257))
            k = int(rng.integers(1, min(8, E) + 1))
        cases.append((T, E, k, method, ng, tg, rsf, 1.0, bool(i % 2)))
    return cases


RANDOM_ROUTE_CASES = _random_route_cases(40, 77)


@pytest.mark.parametrize("case", ROUTE_CASES + RANDOM_ROUTE_CASES,
                         ids=lambda c: f"T{c[0]}E{c[1]}k{c[2]}m{c[3]}g{c[4]}-{c[5]}{'-int' if c[8] else ''}")
def test_route_parity(moe, case):
    T, E, k, method, ng, tg, rsf, scale, int_logits = case
    g = torch.Generator().manual_seed(11)
    if int_logits:
        logits = torch.randint(-2, 3, (T, E), generator=g).float()
    else:
        logits = torch.randn(T, E, generator=g) * scale
    bias = torch.randn(E, generator=g) * 0.1 if method in (DEEPSEEKV3, MINIMAX2) else None
    ids, sc = moe.moe_route(logits.cuda(), method, k, bias=None if bias is None else bias.cuda(),
                            n_group=ng, topk_group=tg, routed_scaling_factor=rsf)
    ids_ref, sc_ref = oracle.route(logits.numpy(), method, k,
                                   bias=None if bias is None else bias.numpy(), n_group=ng,
                                   topk_group=tg, routed_scaling_factor=rsf)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(sc.cpu().numpy(), sc_ref, rtol=1e-6, atol=0)


@pytest.mark.parametrize("method,E,ng,tg", [(DEEPSEEKV3, 256, 8, 4), (MINIMAX2, 128, 1, 1),
                                            (GROUPED_TOPK, 256, 8, 4)])
def test_route_near_ties_in_biased_keys(moe, method, E, ng, tg):
    """Keys that differ by about one fp32 ulp, where the fp32 approximation of the keys
    cannot decide the order: the ids must still match the exact-key oracle."""
    g = torch.Generator().manual_seed(21)
    T = 256
    logits = torch.randn(T, E, generator=g)
    # every other expert gets the next fp32 logit above its neighbour's
    logits[:, 1::2] = torch.nextafter(logits[:, 0::2], torch.full_like(logits[:, 0::2], 10.0))
    bias = None if method == GROUPED_TOPK else torch.zeros(E)
    ids, sc = moe.moe_route(logits.cuda(), method, 8, bias=None if bias is None else bias.cuda(),
                            n_group=ng, topk_group=tg)
    ids_ref, sc_ref = oracle.route(logits.numpy(), method, 8,
                                   bias=None if bias is None else bias.numpy(), n_group=ng,
                                   topk_group=tg)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(sc.cpu().numpy(), sc_ref, rtol=1e-6, atol=0)


def test_route_nonfinite_logits_never_beat_finite(moe):
    logits = torch.randn(32, 16)
    logits[:, 3] = float("nan")
    logits[:, 5] = float("inf")
    logits[:, 7] = -float("inf")
    ids, _ = moe.moe_route(logits.cuda(), RENORMALIZE_NAIVE, 4)
    ids_ref, _ = oracle.route(logits.numpy(), RENORMALIZE_NAIVE, 4)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert not np.isin(ids.cpu().numpy(), [3, 5, 7]).any()


def test_grouped_topk_nonfinite_logits(moe):
    """Non-finite logits count as -inf (score 0) in the grouped top-k as well: they lower
    their group's total and are chosen only when a kept group has nothing better."""
    g = torch.Generator().manual_seed(31)
    logits = torch.randn(40, 32, generator=g)
    logits[:, 1] = float("nan")
    logits[:, 9] = float("inf")
    logits[:, 17] = -float("inf")
    logits[5, 24:28] = -float("inf")       # a whole group without a finite logit
    ids, sc = moe.moe_route(logits.cuda(), GROUPED_TOPK, 4, n_group=8, topk_group=2)
    ids_ref, sc_ref = oracle.route(logits.numpy(), GROUPED_TOPK, 4, n_group=8, topk_group=2)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(sc.cpu().numpy(), sc_ref, rtol=1e-6, atol=0)


# ------------------------------------------------------------------------ permute

@pytest.mark.parametrize("T,E,k", [(300, 8, 2), (5000, 64, 4), (1, 4, 1), (2048, 256, 8), (513, 16, 2),
                                   (9000, 3, 3), (1000, 64, 2)])
def test_permute_parity(moe, T, E, k):
    g = torch.Generator().manual_seed(T + E)
    ids = torch.randint(0, E, (T, k), generator=g, dtype=torch.int32)
    H, I = 384, 192
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    p = moe.make_problem(T, H, I, E, k)
    ws = moe.alloc_workspace(p)
    moe.moe_permute(p, x.cuda(), ids.cuda(), ws)
    torch.cuda.synchronize()
    counts, offsets, perm_src, perm_inv = oracle.permute(ids.numpy(), E)
    P = T * k
    assert np.array_equal(ws.region("counts", E, torch.int32).cpu().numpy(), counts)
    assert np.array_equal(ws.region("offsets", E + 1, torch.int32).cpu().numpy(), offsets)
    assert np.array_equal(ws.region("perm_src", P, torch.int32).cpu().numpy(), perm_src)
    assert np.array_equal(ws.region("perm_inv", P, torch.int32).cpu().numpy(), perm_inv)
    xp = ws.region("x_perm", P * H, torch.bfloat16).view(P, H).cpu()
    assert torch.equal(xp, x[torch.from_numpy(perm_src).long() // k])
    # work lists. Channel tiles: FC1 ceil(I / 128) = 2, FC2 ceil(H / 256) = 2; narrow ones
    # (64 and 128 channels) ceil(I / 64) = 3 and ceil(H / 128) = 3. When T * k >= 256 * E
    # the CTA-pair kernel takes every group: floor(m / 256) + (m % 256 > 0) units per
    # channel tile. Otherwise every group goes to the single-SM list: when T * k <= 32 * E,
    # one narrow tile per narrow channel tile if 1 <= m <= 32; else ceil(m / 128) tiles per
    # channel tile.
    big = (counts >= 1) & (T * k >= 256 * E)
    pair_units = np.where(big, counts // 256 + (counts % 256 > 0), 0)
    row_tiles = counts // 128 + (counts % 128 > 0)
    narrow = ~big & (T * k <= 32 * E) & (counts >= 1) & (counts <= 32)
    for name, wide_c, narrow_c in (("tile_off1", 2, 3), ("tile_off2", 2, 3)):
        single_tiles = np.where(big, 0, np.where(narrow, narrow_c, row_tiles * wide_c))
        lst = ws.region(name, 2 * (E + 1), torch.int32).cpu().numpy()
        assert np.array_equal(lst[:E + 1], np.concatenate([[0], np.cumsum(pair_units * wide_c)]))
        assert np.array_equal(lst[E + 1:], np.concatenate([[0], np.cumsum(single_tiles)]))
    st, flags = moe.moe_read_device_status(ws)
    assert st == moe.MOE_OK and flags == 0


# ------------------------------------------------------------------------ forward (small)

@pytest.mark.parametrize("T", [300, 2500])   # row-by-row copy below 2048 tokens, token-major at and above
def test_permute_rows_with_shared_expert_and_invalid_ids(moe, T):
    """x_perm byte for byte with a shared expert (its rows P + t hold x[t]) and two slots
    whose ids are out of range (no row, perm_inv = -1, status flagged), in both row-copy
    forms of the permute step."""
    E, k, H, I, sI = 16, 4, 256, 128, 128
    g = torch.Generator().manual_seed(T)
    ids = torch.randint(0, E, (T, k), generator=g, dtype=torch.int32)
    ids[5, 1] = E
    ids[T - 1, 0] = -3
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    p = moe.make_problem(T, H, I, E, k, sI)
    ws = moe.alloc_workspace(p)
    moe.moe_permute(p, x.cuda(), ids.cuda(), ws)
    torch.cuda.synchronize()
    flat = ids.numpy().reshape(-1)
    valid = (flat >= 0) & (flat < E)
    # Invalid slots as a sentinel expert E that sorts after every real one: the first n
    # rows of the oracle's permutation are then the valid rows in their stable order.
    _, _, perm_src, _ = oracle.permute(np.where(valid, flat, E).reshape(T, k), E + 1)
    n, P = int(valid.sum()), T * k
    xp = ws.region("x_perm", (P + T) * H, torch.bfloat16).view(P + T, H).cpu()
    assert torch.equal(xp[:n], x[torch.from_numpy(perm_src[:n]).long() // k])
    assert torch.equal(xp[P:], x)
    pinv = ws.region("perm_inv", P, torch.int32).cpu().numpy()
    assert pinv[5 * k + 1] == -1 and pinv[(T - 1) * k] == -1
    st, flags = moe.moe_read_device_status(ws)
    assert st == moe.MOE_ERR_DEVICE_BAD_ID and flags & moe.MOE_DEVICE_FLAG_BAD_ID


def _random_case(T, H, I, E, k, shared_I=0, seed=0, ids_mode="route", method=RENORMALIZE_NAIVE):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=g)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    w13 = (torch.randn(E, 2 * I, H, generator=g) * H ** -0.5).to(torch.bfloat16)
    w2 = (torch.randn(E, H, I, generator=g) * I ** -0.5).to(torch.bfloat16)
    w13s = w2s = None
    if shared_I:
        w13s = (torch.randn(2 * shared_I, H, generator=g) * H ** -0.5).to(torch.bfloat16)
        w2s = (torch.randn(H, shared_I, generator=g) * shared_I ** -0.5).to(torch.bfloat16)
    if ids_mode == "route":
        ids, sc = oracle.route(logits.numpy(), method, k)
    elif ids_mode == "one_expert":
        ids = np.zeros((T, k), np.int32)
        for j in range(k):
            ids[:, j] = j
        sc = np.full((T, k), 1.0 / k)
    elif ids_mode == "random_dup":
        ids = torch.randint(0, E, (T, k), generator=g).numpy().astype(np.int32)
        sc = torch.rand(T, k, generator=g).numpy().astype(np.float64)
    else:
        raise ValueError(ids_mode)
    return dict(x=x, w13=w13, w2=w2, w13s=w13s, w2s=w2s, ids=ids.astype(np.int32),
                sc=sc.astype(np.float32))


def _run_forward_steps(moe, c):
    T, H = c["x"].shape
    E, twoI, _ = c["w13"].shape
    k = c["ids"].shape[1]
    sI = 0 if c["w13s"] is None else c["w13s"].shape[0] // 2
    p = moe.make_problem(T, H, twoI // 2, E, k, sI)
    ws = moe.alloc_workspace(p)
    dev = {n: (None if v is None else (torch.from_numpy(v) if isinstance(v, np.ndarray) else v).cuda())
           for n, v in c.items()}
    y = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    moe.moe_permute(p, dev["x"], dev["ids"], ws)
    moe.moe_fc1(p, dev["w13"], dev["w13s"], ws)
    moe.moe_fc2(p, dev["w2"], dev["w2s"], ws)
    moe.moe_finalize(p, dev["sc"], y, ws)
    torch.cuda.synchronize()
    return p, ws, y, dev


SMALL_CASES = [
    # T, H, I, E, k, shared_I, ids_mode
    (300, 256, 192, 8, 2, 0, "route"),         # weight-major tiles, ragged FC1 channel tile
    (700, 384, 320, 4, 2, 0, "route"),         # token-major + remainder tiles, ragged FC2 tile
    (1000, 256, 256, 8, 1, 0, "one_expert"),   # one expert holds every row (7 full tiles + 104)
    (1100, 256, 256, 4, 1, 0, "one_expert"),   # CTA pairs: 4 units + 76 rows (weight-major)
    (1200, 384, 320, 4, 1, 0, "one_expert"),   # CTA pairs: 4 units + 176 rows (masked pair)
    (1034, 256, 192, 4, 1, 0, "one_expert"),   # CTA pairs: 4 units + 10 rows (64-row X box, 8 used)
    (1100, 192, 192, 4, 1, 0, "one_expert"),   # CTA pairs, 3 K blocks in FC1 and FC2: a stage
                                               # holding one block at the end of every unit
    (150, 256, 192, 4, 1, 0, "one_expert"),    # single-SM: 1 full tile + 22 rows (16-row X boxes)
    (180, 256, 192, 4, 1, 0, "one_expert"),    # single-SM: 1 full tile + 52 rows (64-row X box)
    (300, 128, 64, 2, 1, 0, "one_expert"),     # single-SM: 2 full tiles + 44 rows; FC1's one
                                               # channel tile half past I = 64
    (2200, 256, 192, 4, 2, 256, "route"),      # CTA pairs for routed and shared groups
    # CTA-pair weight-major leftover units of 1, 16, 32, 33 and 128 rows beside full units
    (640, 512, 320, 2, 2, 0, "one_expert"),    # 2 full units + 128 rows, ragged FC1 tile
    (528, 512, 320, 2, 2, 0, "one_expert"),    # 2 full units + 16 rows, ragged FC1 tile
    (272, 256, 192, 1, 1, 0, "one_expert"),    # 1 full unit + 16 rows
    (513, 256, 192, 1, 1, 0, "one_expert"),    # 2 full units + 1 row
    (288, 256, 192, 1, 1, 0, "one_expert"),    # 1 full unit + 32 rows
    (289, 256, 192, 1, 1, 0, "one_expert"),    # 1 full unit + 33 rows
    (2100, 256, 192, 4, 2, 256, "route"),      # routed groups of ~1050 rows, shared 8 full + 52
    (513, 128, 128, 8, 8, 0, "route"),         # k = E: every expert every token
    (200, 192, 128, 16, 4, 128, "random_dup"), # repeated ids in a row, shared expert
    (130, 128, 64, 1, 1, 0, "route"),          # E = 1, k = 1: the dense FFN (128 + 2 rows)
    (1, 128, 128, 8, 2, 0, "route"),           # a single token
    (64, 256, 128, 32, 4, 192, "route"),       # shared expert wider than the routed ones
    (96, 128, 256, 8, 2, 64, "route"),         # shared expert narrower than the routed ones
    (48, 192, 320, 16, 4, 0, "route"),         # narrow tiles: odd K blocks, ragged FC2 tile
    (24, 192, 128, 16, 2, 192, "route"),       # narrow shared expert (odd FC2 K blocks)
]


def _random_cases(n, seed):
    """Seeded random shapes inside the envelope: H and I multiples of 64 up to 512, up to
    64 experts, k up to 8, up to 1200 tokens, with and without a shared expert, each with
    routed, duplicated-random or single-expert ids. Together they land on every GEMM form
    (CTA pairs, single-SM tiles, narrow tiles) with ragged group sizes."""
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        H = 64 * int(rng.integers(1, 9))
        I = 64 * int(rng.integers(1, 9))
        E = int(rng.choice([1, 2, 3, 5, 8, 16, 33, 64]))
        mode = str(rng.choice(["route", "route", "random_dup", "one_expert"]))
        k = int(rng.integers(1, (min(8, E) if mode != "random_dup" else 8) + 1))
        T = int(rng.integers(1, 1201))
        sI = int(rng.choice([0, 0, 64, 192]))
        cases.append((T, H, I, E, k, sI, mode))
    return cases


RANDOM_CASES = _random_cases(20, 2026)


@pytest.mark.parametrize("case", SMALL_CASES + RANDOM_CASES,
                         ids=lambda c: "T{}H{}I{}E{}k{}s{}-{}".format(*c))
def test_forward_steps_parity(moe, case):
    T, H, I, E, k, sI, mode = case
    c = _random_case(T, H, I, E, k, sI, seed=T + H, ids_mode=mode)
    p, ws, y, dev = _run_forward_steps(moe, c)
    x64 = _np64(c["x"])
    w13 = _np64(c["w13"])
    w2 = _np64(c["w2"])
    w13s = None if c["w13s"] is None else _np64(c["w13s"])
    w2s = None if c["w2s"] is None else _np64(c["w2s"])
    y_ref, inter = oracle.forward_permuted(x64, c["ids"], c["sc"], w13, w2, w13s, w2s)
    P = T * k
    assert np.array_equal(ws.region("perm_src", P, torch.int32).cpu().numpy(), inter["perm_src"])
    L = ws.layout
    R, Ih = L["rows"], L["h_ld"]
    h = ws.region("h", R * Ih, torch.bfloat16).view(R, Ih).cpu().double().numpy()
    _check_close(h[:P, :I], inter["h"], H_TOL, "FC1+SwiGLU h")
    out = ws.region("out_perm", R * H, torch.bfloat16).view(R, H).cpu().double().numpy()
    _check_close(out[:P], inter["out"], Y_TOL, "FC2 rows")
    if sI:
        hs_ref = oracle.swiglu(x64 @ w13s.T, sI)
        _check_close(h[P:, :sI], hs_ref, H_TOL, "shared FC1")
        _check_close(out[P:], hs_ref @ w2s.T, Y_TOL, "shared FC2")
    _check_close(y.cpu().double().numpy(), y_ref, Y_TOL, "y")
    # FC1 and FC2 in one launch (moe_fc1_fc2, the launch moe_forward runs) write the same
    # h and out_perm bytes as the two separate launches
    h_steps = ws.region("h", R * Ih, torch.bfloat16).clone()
    out_steps = ws.region("out_perm", R * H, torch.bfloat16).clone()
    ws.region("h", R * Ih, torch.bfloat16).fill_(float("nan"))
    ws.region("out_perm", R * H, torch.bfloat16).fill_(float("nan"))
    moe.moe_permute(p, dev["x"], dev["ids"], ws)
    moe.moe_fc1_fc2(p, dev["w13"], dev["w13s"], dev["w2"], dev["w2s"], ws)
    torch.cuda.synchronize()
    h_f = ws.region("h", R * Ih, torch.bfloat16).view(R, Ih)
    h_s = h_steps.view(R, Ih)
    assert torch.equal(h_f[:P, :I].view(torch.int16), h_s[:P, :I].view(torch.int16))
    if sI:
        assert torch.equal(h_f[P:, :sI].view(torch.int16), h_s[P:, :sI].view(torch.int16))
    assert torch.equal(ws.region("out_perm", R * H, torch.bfloat16).view(torch.int16),
                       out_steps.view(torch.int16))
    # moe_forward (one call) gives the same bytes as the four steps
    y2 = moe.moe_forward(dev["x"], dev["ids"], dev["sc"], dev["w13"], dev["w2"], dev["w13s"],
                         dev["w2s"], workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y2, y)


@pytest.mark.parametrize("T,H,I,E,k,sI,cuts", [
    (300, 256, 192, 8, 2, 128, [(0, 3), (3, 8)]),          # single-SM GEMM path
    (2200, 256, 192, 4, 2, 256, [(0, 1), (1, 2), (2, 4)]),  # CTA-pair GEMM path
    (200, 128, 128, 16, 4, 0, [(0, 5), (5, 6), (6, 16)]),   # a one-expert range
])
def test_forward_partial_over_a_partition(moe, T, H, I, E, k, sI, cuts):
    """The expert-parallel seam: each range's y against the oracle's restricted sum, and
    the ranges' y (shared expert in the first) adding up to moe_forward's y."""
    c = _random_case(T, H, I, E, k, sI, seed=T + E)
    dev = {n: (None if v is None else (torch.from_numpy(v) if isinstance(v, np.ndarray) else v).cuda())
           for n, v in c.items()}
    y_full = moe.moe_forward(dev["x"], dev["ids"], dev["sc"], dev["w13"], dev["w2"], dev["w13s"],
                             dev["w2s"])
    x64 = _np64(c["x"])
    total = torch.zeros(T, H, dtype=torch.float32, device="cuda")
    for n, (lo, hi) in enumerate(cuts):
        w13s, w2s = (dev["w13s"], dev["w2s"]) if n == 0 else (None, None)
        y = moe.moe_forward_partial(dev["x"], dev["ids"], dev["sc"], dev["w13"][lo:hi].contiguous(),
                                    dev["w2"][lo:hi].contiguous(), lo, hi, E, w13s, w2s)
        torch.cuda.synchronize()
        ref = oracle.forward_partial(x64, c["ids"], c["sc"], _np64(c["w13"][lo:hi]),
                                     _np64(c["w2"][lo:hi]), lo, hi,
                                     None if w13s is None else _np64(c["w13s"]),
                                     None if w2s is None else _np64(c["w2s"]))
        _check_close(y.cpu().double().numpy(), ref, Y_TOL, f"partial [{lo}, {hi})")
        total += y.float()
    _check_close(total.cpu().double().numpy(), y_full.cpu().double().numpy(), Y_TOL,
                 "sum of the partials vs moe_forward")


GATE_TOL = 1e-4   # fp32 accumulation of H bf16 products, relative to max|logit|


@pytest.mark.parametrize("T,H,E,ns,method", [
    (300, 256, 8, 0, RENORMALIZE_NAIVE),      # one column tile, ragged last row tile
    (513, 1024, 256, 1, DEEPSEEKV3),          # FSE: 257 gate rows -> two column tiles
    (64, 2048, 128, 0, RENORMALIZE_NAIVE),    # decode size: one row tile split along K
    (1, 128, 16, 1, LLAMA4),                  # a single token
    (4096, 4096, 8, 0, RENORMALIZE_NAIVE),    # mixtral_prefill's gate
    (100, 512, 2, 1, RENORMALIZE_NAIVE),      # 3 gate rows (padded to 4), FSE row last
    (77, 256, 15, 1, RENORMALIZE_NAIVE),      # 16 rows, one 16-row MMA tile
    (100, 448, 8, 0, RENORMALIZE_NAIVE),      # 7 K blocks over 2 CTAs: a stage holding one
    (2048, 5120, 16, 1, LLAMA4),              # llama4_scout's gate: 16 clusters of 8 do not
                                              # all fit, the K split drops to 4
])
def test_gate_parity_and_routing_on_its_logits(moe, T, H, E, ns, method):
    g = torch.Generator().manual_seed(T + E)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    wg = (torch.randn(E + ns, H, generator=g) * H ** -0.5).to(torch.bfloat16)
    lg, sg = moe.moe_gate(x.cuda(), wg.cuda(), E)
    lg2, _ = moe.moe_gate(x.cuda(), wg.cuda(), E)
    torch.cuda.synchronize()
    assert torch.equal(lg, lg2)   # fixed reduction order
    ref_r, ref_s = oracle.gate(_np64(x), _np64(wg), E)
    _check_close(lg.cpu().double().numpy(), ref_r, GATE_TOL, "routed logits")
    if ns:
        _check_close(sg.cpu().double().numpy(), ref_s, GATE_TOL, "shared gate logits")
    else:
        assert sg is None
    # The routing decision is taken on the same fp32 logits on both sides.
    k = 1 if method == LLAMA4 else min(8, E)
    kw = dict(n_group=8, topk_group=4, routed_scaling_factor=2.5) if method == DEEPSEEKV3 else {}
    ids, sc = moe.moe_route(lg, method, k, **kw)
    ids_ref, sc_ref = oracle.route(lg.cpu().numpy(), method, k, **kw)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(sc.cpu().numpy(), sc_ref, rtol=1e-6, atol=0)


GATE_ROUTE_CASES = [
    # T, H, E, n_shared, method, k, routing kwargs, integer-valued inputs (exact ties)
    (300, 256, 8, 0, RENORMALIZE_NAIVE, 2, {}, False),
    (513, 1024, 256, 1, DEEPSEEKV3, 8, dict(n_group=8, topk_group=4, routed_scaling_factor=2.5),
     False),                                                   # FSE row in a second column tile
    (64, 2048, 128, 0, RENORMALIZE_NAIVE, 8, {}, False),       # decode: the gate split along K
    (1, 128, 16, 1, LLAMA4, 1, {}, False),                     # a single token
    (4096, 4096, 8, 0, RENORMALIZE_NAIVE, 2, {}, False),       # mixtral_prefill's gate
    (512, 7168, 256, 1, DEEPSEEKV3, 8, dict(n_group=8, topk_group=4, routed_scaling_factor=2.5),
     False),                                                   # dsv3_layer's gate with FSE
    (1000, 512, 64, 0, SIGMOID_RENORM, 4, {}, False),
    (257, 512, 256, 0, GROUPED_TOPK, 8, dict(n_group=8, topk_group=4, routed_scaling_factor=2.5),
     False),
    (200, 256, 96, 0, MINIMAX2, 6, {}, False),
    (100, 512, 33, 0, DEFAULT, 3, {}, False),
    (100, 256, 64, 1, RENORMALIZE, 6, {}, False),
    (300, 128, 16, 0, RENORMALIZE_NAIVE, 4, {}, True),         # integer logits: ties
    (300, 128, 16, 0, DEEPSEEKV3, 4, dict(n_group=4, topk_group=2), True),
    (300, 128, 32, 0, GROUPED_TOPK, 4, dict(n_group=8, topk_group=2), True),
    (2048, 5120, 16, 1, LLAMA4, 1, {}, False),                 # llama4_scout's gate (K split 4)
    (100, 448, 8, 0, RENORMALIZE_NAIVE, 2, {}, False),         # a stage holding one K block
]


@pytest.mark.parametrize("case", GATE_ROUTE_CASES,
                         ids=lambda c: "T{}H{}E{}s{}m{}k{}{}".format(*c[:6], "-int" if c[7] else ""))
def test_gate_route_fused(moe, case):
    """The gate with routing fused into its epilogue: the logits it writes equal moe_gate's,
    and its ids and scales equal moe_route's on those logits, bit for bit; ids bit-exact and
    scales within 1e-6 against the oracle routing the same fp32 logits."""
    T, H, E, ns, method, k, kw, ints = case
    g = torch.Generator().manual_seed(T + H + E)
    if ints:   # entries in {-1, 0, 1}: every logit an exact integer
        x = torch.randint(-1, 2, (T, H), generator=g).to(torch.bfloat16).cuda()
        wg = torch.randint(-1, 2, (E + ns, H), generator=g).to(torch.bfloat16).cuda()
    else:
        x = torch.randn(T, H, generator=g).to(torch.bfloat16).cuda()
        wg = (torch.randn(E + ns, H, generator=g) * H ** -0.5).to(torch.bfloat16).cuda()
    bias = (torch.randn(E, generator=g) * 0.1).cuda() if method in (DEEPSEEKV3, MINIMAX2) else None
    lg, sg = moe.moe_gate(x, wg, E)
    ids, sc, lg2, sg2 = moe.moe_gate_route(x, wg, method, k, E, bias=bias, want_logits=True, **kw)
    ids3, sc3, lg3, _ = moe.moe_gate_route(x, wg, method, k, E, bias=bias, **kw)
    torch.cuda.synchronize()
    assert lg3 is None
    assert torch.equal(lg2, lg)
    if ns:
        assert torch.equal(sg2, sg)
    ids_r, sc_r = moe.moe_route(lg, method, k, bias=bias, **kw)
    assert torch.equal(ids, ids_r)
    assert torch.equal(sc.view(torch.int32), sc_r.view(torch.int32))
    assert torch.equal(ids3, ids) and torch.equal(sc3, sc)
    ids_ref, sc_ref = oracle.route(lg.cpu().numpy(), method, k,
                                   bias=None if bias is None else bias.cpu().numpy(), **kw)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(sc.cpu().numpy(), sc_ref, rtol=1e-6, atol=0)


def _random_gate_cases(n, seed):
    """Seeded random gate problems: T up to 2500, H up to 3072, the routing problems of
    _random_route_cases, with or without the shared expert's gate row."""
    rng = np.random.default_rng(seed)
    cases = []
    for (_, E, k, method, ng, tg, rsf, _, _) in _random_route_cases(n, seed + 1):
        T = int(rng.integers(1, 2501))
        H = 64 * int(rng.integers(1, 49))
        ns = int(rng.integers(0, 2))
        kw = {} if method not in (DEEPSEEKV3, GROUPED_TOPK) else dict(
            n_group=ng, topk_group=tg, routed_scaling_factor=rsf)
        cases.append((T, H, E, ns, method, k, kw))
    return cases


@pytest.mark.parametrize("case", _random_gate_cases(16, 303),
                         ids=lambda c: "T{}H{}E{}s{}m{}k{}".format(*c[:6]))
def test_gate_random_shapes(moe, case):
    """Random gate shapes (K split, cluster size, stage grouping and column tiles vary with
    them): the logits against the oracle's gate, the fused routing against the route
    kernel on those logits bit for bit, and ids bit-exact against the oracle."""
    T, H, E, ns, method, k, kw = case
    g = torch.Generator().manual_seed(T * 7 + H + E)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    wg = (torch.randn(E + ns, H, generator=g) * H ** -0.5).to(torch.bfloat16)
    bias = (torch.randn(E, generator=g) * 0.1).cuda() if method in (DEEPSEEKV3, MINIMAX2) else None
    lg, sg = moe.moe_gate(x.cuda(), wg.cuda(), E)
    ids, sc, _, _ = moe.moe_gate_route(x.cuda(), wg.cuda(), method, k, E, bias=bias, **kw)
    torch.cuda.synchronize()
    ref_r, ref_s = oracle.gate(_np64(x), _np64(wg), E)
    _check_close(lg.cpu().double().numpy(), ref_r, GATE_TOL, "routed logits")
    if ns:
        _check_close(sg.cpu().double().numpy(), ref_s, GATE_TOL, "shared gate logits")
    ids_r, sc_r = moe.moe_route(lg, method, k, bias=bias, **kw)
    assert torch.equal(ids, ids_r)
    assert torch.equal(sc.view(torch.int32), sc_r.view(torch.int32))
    ids_ref, sc_ref = oracle.route(lg.cpu().numpy(), method, k,
                                   bias=None if bias is None else bias.cpu().numpy(), **kw)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(sc.cpu().numpy(), sc_ref, rtol=1e-6, atol=0)


def test_forward_with_the_fused_shared_gate(moe):
    T, H, I, E, k, sI = 300, 256, 192, 8, 2, 128
    c = _random_case(T, H, I, E, k, sI, seed=5)
    dev = {n: (None if v is None else (torch.from_numpy(v) if isinstance(v, np.ndarray) else v).cuda())
           for n, v in c.items()}
    sg = torch.randn(T, generator=torch.Generator().manual_seed(6)) * 2.0
    y = moe.moe_forward_partial(dev["x"], dev["ids"], dev["sc"], dev["w13"], dev["w2"], 0, E, E,
                                dev["w13s"], dev["w2s"], shared_gate=sg.cuda())
    torch.cuda.synchronize()
    ref = oracle.forward(_np64(c["x"]), c["ids"], c["sc"], ExpertView(c["w13"]),
                         ExpertView(c["w2"]), _np64(c["w13s"]), _np64(c["w2s"]),
                         shared_gate=sg.double().numpy())
    _check_close(y.cpu().double().numpy(), ref, Y_TOL, "y with the shared gate")


@pytest.mark.parametrize("T,E,k", [(65536, 8, 8), (40000, 256, 8)])
def test_largest_row_counts(moe, T, E, k):
    """Many permuted rows (T*k up to 524,288): routing, the permutation and y on every
    token."""
    H, I = 128, 64
    g = torch.Generator(device="cuda").manual_seed(T)
    logits = torch.randn(T, E, generator=g, device="cuda")
    x = torch.randn(T, H, generator=g, device="cuda").to(torch.bfloat16)
    w13 = (torch.randn(E, 2 * I, H, generator=g, device="cuda") * H ** -0.5).to(torch.bfloat16)
    w2 = (torch.randn(E, H, I, generator=g, device="cuda") * I ** -0.5).to(torch.bfloat16)
    ids, sc = moe.moe_route(logits, RENORMALIZE_NAIVE, k)
    p = moe.make_problem(T, H, I, E, k)
    ws = moe.alloc_workspace(p)
    y = moe.moe_forward(x, ids, sc, w13, w2, workspace=ws)
    torch.cuda.synchronize()
    ids_ref, sc_ref = oracle.route(logits.cpu().numpy(), RENORMALIZE_NAIVE, k)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    counts, offsets, perm_src, perm_inv = oracle.permute(ids_ref, E)
    assert np.array_equal(ws.region("perm_src", T * k, torch.int32).cpu().numpy(), perm_src)
    y_ref = oracle.forward(x.cpu().double().numpy(), ids_ref, sc_ref, ExpertView(w13),
                           ExpertView(w2))
    _check_close(y.cpu().double().numpy(), y_ref, Y_TOL, "y (every token)")
    st, flags = moe.moe_read_device_status(ws)
    assert st == moe.MOE_OK and flags == 0


def test_forward_is_deterministic(moe):
    c = _random_case(2000, 256, 256, 16, 4, 0, seed=3)
    _, ws, y1, dev = _run_forward_steps(moe, c)
    perm1 = ws.region("perm_src", 8000, torch.int32).clone()
    y2 = moe.moe_forward(dev["x"], dev["ids"], dev["sc"], dev["w13"], dev["w2"], workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    assert torch.equal(perm1, ws.region("perm_src", 8000, torch.int32))


def test_bad_ids_are_skipped_and_flagged(moe):
    c = _random_case(64, 128, 128, 8, 2, 0, seed=5, ids_mode="random_dup")
    ids = c["ids"].copy()
    ids[3, 1] = 8
    ids[10, 0] = -1
    c["ids"] = ids
    p, ws, y, dev = _run_forward_steps(moe, c)
    st, flags = moe.moe_read_device_status(ws)
    assert st == moe.MOE_ERR_DEVICE_BAD_ID and flags & moe.MOE_DEVICE_FLAG_BAD_ID
    assert moe.moe_read_device_status(ws)[0] == moe.MOE_OK   # the read cleared it
    sc = c["sc"].copy()
    sc[3, 1] = 0
    sc[10, 0] = 0
    ids_ok = np.where(ids < 0, 0, np.where(ids >= 8, 0, ids))
    y_ref = oracle.forward(_np64(c["x"]), ids_ok, sc, _np64(c["w13"]), _np64(c["w2"]))
    _check_close(y.cpu().double().numpy(), y_ref, Y_TOL, "y with skipped rows")
    pinv = ws.region("perm_inv", 128, torch.int32).cpu().numpy()
    assert pinv[3 * 2 + 1] == -1 and pinv[10 * 2 + 0] == -1


def test_device_wait_timeout_is_reported_and_the_context_stays_usable(moe):
    """The failure path without a fault: a pipeline wait that nothing completes runs out
    after the kernels' 2 s limit, the host reads MOE_DEVICE_FLAG_TIMEOUT, the other role
    (which would have waited until 3 s) is released by the abort flag, and a forward on
    the same context afterwards is correct and reports no error."""
    import time
    c = _random_case(64, 128, 128, 8, 2, 0, seed=7)
    p, ws, y0, dev = _run_forward_steps(moe, c)
    assert moe.moe_read_device_status(ws)[0] == moe.MOE_OK
    t0 = time.perf_counter()
    moe.moe_selftest_wait(ws)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    released = int(ws.region("status", 4, torch.int32)[1].item())
    st, flags = moe.moe_read_device_status(ws)
    assert st == moe.MOE_ERR_DEVICE_TIMEOUT and flags & moe.MOE_DEVICE_FLAG_TIMEOUT
    assert released == 1, "the consumer waited out its own limit: the abort flag did not reach it"
    assert 1.5 < dt < 2.8, dt
    y = torch.empty_like(y0)
    moe.moe_permute(p, dev["x"], dev["ids"], ws)
    moe.moe_fc1(p, dev["w13"], None, ws)
    moe.moe_fc2(p, dev["w2"], None, ws)
    moe.moe_finalize(p, dev["sc"], y, ws)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws)[0] == moe.MOE_OK
    assert torch.equal(y, y0)
    y_ref = oracle.forward(_np64(c["x"]), c["ids"], c["sc"], _np64(c["w13"]), _np64(c["w2"]))
    _check_close(y.cpu().double().numpy(), y_ref, Y_TOL, "y after the self-test")


_THREADED_SCRIPT = r"""
import sys, threading, torch
import mixture_experts_layer_03_gb300 as moe
shapes = [  # T, H, I, E, k, shared_I: single-SM, narrow, CTA-pair, shared-expert launches
    (300, 256, 192, 8, 2, 0), (48, 192, 320, 16, 4, 0), (2200, 256, 192, 4, 2, 256),
    (64, 256, 128, 32, 4, 192), (513, 128, 128, 8, 8, 0), (1, 128, 128, 8, 2, 0)]
g = torch.Generator().manual_seed(3)
cases = []
for T, H, I, E, k, sI in shapes:
    c = dict(x=torch.randn(T, H, generator=g).to(torch.bfloat16),
             ids=torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).int(),
             sc=torch.rand(T, k, generator=g),
             w13=(torch.randn(E, 2 * I, H, generator=g) * H ** -0.5).to(torch.bfloat16),
             w2=(torch.randn(E, H, I, generator=g) * I ** -0.5).to(torch.bfloat16),
             w13s=(torch.randn(2 * sI, H, generator=g) * H ** -0.5).to(torch.bfloat16) if sI else None,
             w2s=(torch.randn(H, sI, generator=g) * sI ** -0.5).to(torch.bfloat16) if sI else None)
    cases.append({n: (None if v is None else v.cuda()) for n, v in c.items()})
torch.cuda.synchronize()

def run(c, stream=None):
    return moe.moe_forward(c["x"], c["ids"], c["sc"], c["w13"], c["w2"], c["w13s"], c["w2s"],
                           stream=stream)

out, err = [None] * len(cases), []
start = threading.Barrier(len(cases))
def worker(i):
    try:
        s = torch.cuda.Stream()
        start.wait()                      # every thread's first call at the same moment
        with torch.cuda.stream(s):
            y = run(cases[i], s)
        s.synchronize()
        out[i] = y
    except Exception as e:
        err.append(repr(e))
ts = [threading.Thread(target=worker, args=(i,)) for i in range(len(cases))]
for t in ts: t.start()
for t in ts: t.join()
assert not err, err
for i, c in enumerate(cases):
    y = run(c)
    torch.cuda.synchronize()
    assert torch.equal(y, out[i]), f"case {i}: threaded result differs"
print("threaded-ok")
"""


def test_concurrent_calls_from_host_threads_in_a_fresh_process():
    """The library's one-time per-device setup and its launches from several host threads
    at once (each thread: its own stream and workspace, first use in a fresh process)
    give the same bytes as the same forwards run one after another."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _THREADED_SCRIPT], cwd=root, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "threaded-ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]


def test_zero_tokens_is_a_noop(moe):
    x = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(0, 2, dtype=torch.int32, device="cuda")
    sc = torch.empty(0, 2, dtype=torch.float32, device="cuda")
    w13 = torch.zeros(4, 128, 128, dtype=torch.bfloat16, device="cuda")
    w2 = torch.zeros(4, 128, 64, dtype=torch.bfloat16, device="cuda")
    y = moe.moe_forward(x, ids, sc, w13, w2)
    assert y.shape == (0, 128)
    i, s = moe.moe_route(torch.empty(0, 8, device="cuda"), RENORMALIZE_NAIVE, 2)
    assert i.shape == (0, 2)


def test_cast_is_round_to_nearest_even(moe):
    v = torch.randn(100003) * 10
    v[:4] = torch.tensor([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -0.0, float("inf")])
    got = moe.moe_cast_f32_to_bf16(v.cuda()).cpu()
    assert torch.equal(got.view(torch.int16), v.to(torch.bfloat16).view(torch.int16))


# ------------------------------------------------------------------------ full-size workloads

def _leftover_rows(offsets, unit):
    """Permuted rows past each expert's last full unit of `unit` rows (the rows the GEMMs
    cover with their partial, weight-major or masked units)."""
    rows = []
    for e in range(len(offsets) - 1):
        a, b = int(offsets[e]), int(offsets[e + 1])
        rem = (b - a) % unit
        if rem:
            rows.append(np.arange(b - rem, b))
    return np.concatenate(rows) if rows else np.zeros(0, np.int64)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["tiny", "mixtral_prefill", "qwen3_decode", "dsv3_layer", "skewed",
                                  "llama4_scout", "minimax_m2"])
def test_workload_full_size(moe, name):
    """The workloads at full size, in the launch configuration the bench times
    (moe_route then moe_forward on one stream). Routing, counts and the permutation are
    checked on every token; y on every token, and the intermediate h (FC1 + SwiGLU) and
    out_perm (FC2) rows on every permuted row, against the oracle's five-step forward.
    The rows of each expert past its last full 256-row unit are named separately (the
    GEMMs' partial units)."""
    w: Workload = WORKLOADS[name]
    inp = make_inputs(w, device="cuda", seed=0)
    if w.in_dtype == "f32":
        x = moe.moe_cast_f32_to_bf16(inp["x"])
        w13 = moe.moe_cast_f32_to_bf16(inp["w13"])
        w2 = moe.moe_cast_f32_to_bf16(inp["w2"])
    else:
        x, w13, w2 = inp["x"], inp["w13"], inp["w2"]
    w13s, w2s = inp["w13_s"], inp["w2_s"]
    p = moe.make_problem(w.T, w.H, w.I, w.E, w.k, w.shared_I)
    ws = moe.alloc_workspace(p)
    ids, sc = moe.moe_route(inp["logits"], w.method, w.k, bias=inp["bias"], n_group=w.n_group,
                            topk_group=w.topk_group, routed_scaling_factor=w.rsf)
    y = moe.moe_forward(x, ids, sc, w13, w2, w13s, w2s, workspace=ws)
    torch.cuda.synchronize()

    logits = inp["logits"].cpu().numpy()
    bias = None if inp["bias"] is None else inp["bias"].cpu().numpy()
    ids_ref, sc_ref = oracle.route(logits, w.method, w.k, bias=bias, n_group=w.n_group,
                                   topk_group=w.topk_group, routed_scaling_factor=w.rsf)
    ids_gpu = ids.cpu().numpy()
    mism = np.argwhere((ids_gpu != ids_ref).any(1)).ravel()
    assert mism.size == 0, f"{name}: ids differ on tokens {mism[:10]}"
    np.testing.assert_allclose(sc.cpu().numpy(), sc_ref, rtol=1e-6, atol=0)
    counts, offsets, perm_src, perm_inv = oracle.permute(ids_ref, w.E)
    assert np.array_equal(ws.region("counts", w.E, torch.int32).cpu().numpy(), counts)
    assert np.array_equal(ws.region("perm_src", w.P, torch.int32).cpu().numpy(), perm_src)
    assert np.array_equal(ws.region("perm_inv", w.P, torch.int32).cpu().numpy(), perm_inv)
    st, flags = moe.moe_read_device_status(ws)
    assert st == moe.MOE_OK and flags == 0
    assert torch.isfinite(y.float()).all()

    if w.in_dtype == "f32":   # the oracle takes the fp32 originals (the cast counts as error)
        X = inp["x"].cpu().double().numpy()
        W13, W2 = ExpertView(inp["w13"]), ExpertView(inp["w2"])
        W13s = W2s = None
    else:
        X = x.cpu().double().numpy()
        W13, W2 = ExpertView(w13), ExpertView(w2)
        W13s = None if w13s is None else _np64(w13s)
        W2s = None if w2s is None else _np64(w2s)
    # the oracle's weights are the oracle's own (fp64) scales, so the y comparison also
    # carries the fp32 rounding of the device's scales
    y_ref, inter = oracle.forward_permuted(X, ids_ref, sc_ref, W13, W2, W13s, W2s)
    _check_close(y.cpu().double().numpy(), y_ref, Y_TOL, f"{name} y (every token)")

    L = ws.layout
    R, Ih = L["rows"], L["h_ld"]
    P = w.P
    h_ref, out_ref = inter["h"], inter["out"]
    h_gpu = ws.region("h", R * Ih, torch.bfloat16).view(R, Ih)[:P, :w.I].cpu().double().numpy()
    _check_close(h_gpu, h_ref, H_TOL, f"{name} h (every permuted row)")
    out_gpu = ws.region("out_perm", R * w.H, torch.bfloat16).view(R, w.H).cpu().double().numpy()
    _check_close(out_gpu[:P], out_ref, Y_TOL, f"{name} out_perm (every permuted row)")
    left = _leftover_rows(offsets, 256)
    if left.size:
        hb = H_TOL * np.abs(h_ref).max()
        ob = Y_TOL * np.abs(out_ref).max()
        eh = np.abs(h_gpu[left] - h_ref[left]).max()
        eo = np.abs(out_gpu[left] - out_ref[left]).max()
        assert eh <= hb, f"{name} h on the {left.size} leftover rows: {eh:.4e} > {hb:.4e}"
        assert eo <= ob, f"{name} out_perm on the {left.size} leftover rows: {eo:.4e} > {ob:.4e}"
    if w.shared_I:
        hs_ref = oracle.swiglu(X @ W13s.T, w.shared_I)
        hs_gpu = ws.region("h", R * Ih, torch.bfloat16).view(R, Ih)[P:, :w.shared_I]
        _check_close(hs_gpu.cpu().double().numpy(), hs_ref, H_TOL, f"{name} shared h")
        _check_close(out_gpu[P:], hs_ref @ W2s.T, Y_TOL, f"{name} shared out_perm rows")

"""Pins for the oracle: values the pages print, closed forms, special cases,
brute force and invariants.  CPU only."""
import itertools
import json
import math
import os

import numpy as np
import pytest
from scipy import stats

from oracle import dspark_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- survival / STS

def test_survival_table_from_page():
    g = _gold("survival_table.json")
    c = np.array([g["c"]], dtype=np.float32)
    a = O.prefix_survival(c)[0]
    printed = np.array(g["a_printed"])
    assert np.all(np.abs(a - printed) <= 1e-3 + 1e-7)
    # exact product at position 4 and the page's chained 3-decimal rounding
    assert abs(float(a[3]) - 0.96 * 0.93 * 0.86 * 0.70) < 1e-6
    chained, acc = [], None
    for ci in g["c"]:
        acc = ci if acc is None else round(acc * ci, 3)
        chained.append(round(acc, 3))
    assert chained == g["a_printed"]


def test_survival_is_running_product_in_fp32_order():
    rng = np.random.default_rng(1)
    c = rng.uniform(0.3, 1.0, size=(5, 9)).astype(np.float32)
    a = O.prefix_survival(c)
    for r in range(5):
        acc = np.float32(1.0)
        for j in range(9):
            acc = np.float32(acc * c[r, j]) if j else c[r, 0]
            assert a[r, j] == acc
    assert np.all(np.diff(a, axis=1) <= 0)


def test_sts_unit_temperature_is_identity():
    rng = np.random.default_rng(2)
    a = np.sort(rng.uniform(0.01, 0.99, size=(4, 8)).astype(np.float32), axis=1)[:, ::-1].copy()
    ah = O.sts_calibrate(a, np.ones(8, dtype=np.float32))
    # sigmoid(logit(a)) = a up to one fp32 rounding of the fp64 result
    assert np.all(np.abs(ah.astype(np.float64) - a.astype(np.float64)) <= 6e-8 * a)


def test_sts_limits_and_textbook_temperature_scaling():
    a = np.array([[0.9, 0.6, 0.3, 0.1]], dtype=np.float32)
    # very hot temperature -> 1/2 ; then clamped non-increasing
    hot = O.sts_calibrate(a, np.full(4, 1e6, dtype=np.float32))
    assert np.all(np.abs(hot - 0.5) < 1e-5)
    # temperature scaling of a binary logit: sigmoid(logit(a)/T) (scipy's expit/logit)
    from scipy.special import expit, logit
    T = np.array([1.0, 1.2, 1.4, 1.6], dtype=np.float32)
    ah = O.sts_calibrate(a, T)
    ref = expit(logit(a.astype(np.float64)) / T.astype(np.float64))
    ref = np.minimum.accumulate(ref.astype(np.float32), axis=1)
    assert np.all(np.abs(ah - ref) <= 1e-7)
    # cold temperature pushes towards 0/1; the clamp keeps a prefix-survival shape
    a2 = np.array([[0.8, 0.7, 0.45, 0.40]], dtype=np.float32)
    ah2 = O.sts_calibrate(a2, np.array([1.0, 1.0, 0.1, 5.0], dtype=np.float32))
    assert np.all(np.diff(ah2[0]) <= 0)


# ---------------------------------------------------------------- greedy scheduler

def _objective(ah, windows, cost, B):
    E = B + sum(float(ah[r, j]) for r in range(B) for j in range(int(windows[r])))
    return E / float(cost[B + int(sum(windows))])


def _cost(theta, n, bias=20.0):
    return (bias + theta * np.arange(n, dtype=np.float64)).astype(np.float32)


@pytest.mark.parametrize("seed", range(12))
def test_greedy_reaches_bruteforce_optimum(seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 4))
    gamma = int(rng.integers(1, 5))
    theta = float(rng.choice([0.02, 0.19, 0.5, 2.0, 6.0]))
    conf = rng.normal(1.0, 1.5, size=(B, gamma)).astype(np.float32)
    temps = np.linspace(1.0, 1.5, gamma).astype(np.float32)
    budget = int(rng.integers(B, B * (gamma + 1) + 1))
    cost = _cost(theta, B * (gamma + 1) + 2)
    s = O.schedule(conf, 1, temps, cost, budget, O.COMPACT)
    best, arg = -1.0, []
    for w in itertools.product(range(gamma + 1), repeat=B):
        if B + sum(w) > budget:
            continue
        v = _objective(s.a_hat, w, cost, B)
        if v > best + 1e-15:
            best, arg = v, [w]
        elif abs(v - best) <= 1e-15:
            arg.append(w)
    got = _objective(s.a_hat, s.windows, cost, B)
    assert got >= best - 1e-12 * best
    if len(arg) == 1 and not s.listed:
        assert tuple(int(x) for x in s.windows) == arg[0]


def test_greedy_identical_requests_round_robin():
    gamma, B = 6, 5
    row = np.array([2.5, 2.0, 1.2, 0.3, -0.5, -1.0], dtype=np.float32)
    conf = np.tile(row, (B, 1))
    s = O.schedule(conf, 1, np.ones(gamma, np.float32), _cost(0.19, 64), 64, O.COMPACT)
    w = s.windows
    assert w.max() - w.min() <= 1
    # equal survival: lower request index first
    assert np.all(np.diff(w) <= 0)


def test_greedy_zero_slope_verifies_everything_within_budget():
    rng = np.random.default_rng(7)
    conf = rng.normal(0.0, 2.0, size=(4, 5)).astype(np.float32)
    s = O.schedule(conf, 1, np.ones(5, np.float32), np.full(40, 20.0, np.float32), 100, O.COMPACT)
    assert np.all(s.windows == 5)
    s2 = O.schedule(conf, 1, np.ones(5, np.float32), np.full(40, 20.0, np.float32), 13, O.COMPACT)
    assert 4 + s2.windows.sum() == 13 and s2.stop_reason == "budget"


def test_greedy_windows_shrink_with_load_and_cost_slope():
    rng = np.random.default_rng(11)
    gamma = 8
    conf = rng.normal(1.5, 1.0, size=(64, gamma)).astype(np.float32)
    temps = np.linspace(1.0, 1.5, gamma).astype(np.float32)
    prev = None
    for theta in (0.01, 0.05, 0.19, 0.5, 2.0):
        s = O.schedule(conf, 1, temps, _cost(theta, 64 * 9 + 2), 10_000, O.COMPACT)
        if prev is not None:
            assert np.all(s.windows <= prev)
        prev = s.windows
    # more concurrent requests -> the first requests' windows do not grow
    prev = None
    for B in (4, 8, 16, 32, 64):
        s = O.schedule(conf[:B], 1, temps, _cost(0.19, 64 * 9 + 2), 10_000, O.COMPACT)
        if prev is not None:
            assert np.all(s.windows[: len(prev)] <= prev)
        prev = s.windows


def test_static_mode_is_whole_block():
    conf = np.zeros((3, 4), np.float32)
    s = O.schedule(conf, 1, np.ones(4, np.float32), _cost(5.0, 20), 8, O.STATIC)
    assert np.all(s.windows == 4) and s.M == 15


# ---------------------------------------------------------------- pack

def test_pack_example_from_page():
    g = _gold("pack_example.json")
    w = np.array(g["windows"], np.int32)
    B = len(w)
    pk = O.pack(w, np.array([10, 20, 30]), np.array([1, 2, 3]), np.arange(B * 6).reshape(B, 6),
                g["tiers"], O.COMPACT, 6)
    assert pk.cu_seqlens.tolist() == g["cu_seqlens"]
    assert pk.M == g["M"] and pk.tier == g["tier"]
    # row contents: anchor then drafts, positions ctx + i, padding marked -1
    assert pk.row_req.tolist() == [0] * 6 + [1] * 4 + [2] * 3 + [-1] * 3
    assert pk.row_pos[:6].tolist() == list(range(10, 16))
    assert pk.row_tok[:6].tolist() == [1, 0, 1, 2, 3, 4]
    assert pk.row_tok[6:10].tolist() == [2, 6, 7, 8]


@pytest.mark.parametrize("mode", [O.COMPACT, O.STATIC, O.CAP_ACCEPT])
def test_pack_invariants(mode):
    rng = np.random.default_rng(5)
    B, gamma = 9, 5
    w = rng.integers(0, gamma + 1, size=B).astype(np.int32)
    if mode == O.STATIC:
        w[:] = gamma
    tiers = [8, 16, 32, 64]
    pk = O.pack(w, rng.integers(0, 100, B), rng.integers(0, 50, B),
                rng.integers(0, 50, (B, gamma)), tiers, mode, gamma)
    n = (w + 1) if mode != O.CAP_ACCEPT else np.full(B, gamma + 1)
    assert pk.M == int(n.sum()) == pk.cu_seqlens[-1]
    assert np.all(np.diff(pk.cu_seqlens) == n)
    bigger = [t for t in tiers if t >= pk.M]
    assert pk.tier == (min(bigger) if bigger else pk.M)
    assert np.all(pk.row_req[pk.M:] == -1)


def test_pack_tier_edges():
    """M equal to a tier takes that tier (no padding); one more row takes the next; M
    above every tier runs unpadded; a single request with w = 0 packs its anchor alone."""
    gamma = 6
    anchor, ctx = np.array([5, 6, 7]), np.array([0, 16, 100])
    drafts = np.arange(3 * gamma).reshape(3, gamma)
    tiers = [4, 9, 16]
    exact = O.pack(np.array([3, 2, 1], np.int32), ctx, anchor, drafts, tiers, O.COMPACT, gamma)
    assert exact.M == 9 and exact.tier == 9 and np.all(exact.row_req >= 0)
    plus1 = O.pack(np.array([3, 2, 2], np.int32), ctx, anchor, drafts, tiers, O.COMPACT, gamma)
    assert plus1.M == 10 and plus1.tier == 16 and plus1.row_req[10:].tolist() == [-1] * 6
    over = O.pack(np.array([6, 6, 6], np.int32), ctx, anchor, drafts, tiers, O.COMPACT, gamma)
    assert over.M == 21 and over.tier == 21
    one = O.pack(np.array([0], np.int32), ctx[:1], anchor[:1], drafts[:1], tiers, O.COMPACT,
                 gamma)
    assert one.cu_seqlens.tolist() == [0, 1] and one.M == 1 and one.tier == 4
    assert one.row_tok.tolist() == [5, -1, -1, -1] and one.row_pos[0] == 0


# ---------------------------------------------------------------- attention

def _toy_gqa(rng, B=2, Hq=4, Hkv=2, D=8, P=4, ctx=(5, 0), n=(3, 2)):
    n_pages = sum((c + P - 1) // P for c in ctx) + 2
    kc = rng.normal(size=(n_pages, P, Hkv, D))
    vc = rng.normal(size=(n_pages, P, Hkv, D))
    perm = rng.permutation(n_pages)
    pt = -np.ones((B, 4), np.int64)
    k = 0
    for r in range(B):
        for p in range((ctx[r] + P - 1) // P):
            pt[r, p] = perm[k]
            k += 1
    cu = np.concatenate([[0], np.cumsum(n)])
    M = int(cu[-1])
    q = rng.normal(size=(M, Hq, D))
    kn = rng.normal(size=(M, Hkv, D))
    vn = rng.normal(size=(M, Hkv, D))
    return dict(q=q, kn=kn, vn=vn, kc=kc, vc=vc, pt=pt, ctx=np.array(ctx), cu=cu)


def _dense_masked_reference(t, Hq, Hkv, scale):
    """Same attention written as one dense masked matrix per request (no paging,
    no per-row prefix concatenation)."""
    from scipy.special import logsumexp, softmax
    B = len(t["ctx"])
    P = t["kc"].shape[1]
    G = Hq // Hkv
    outs, lses = [], []
    for r in range(B):
        c0, c1 = t["cu"][r], t["cu"][r + 1]
        ctx = t["ctx"][r]
        flat_k = np.zeros((ctx + c1 - c0, Hkv, t["kc"].shape[-1]))
        flat_v = np.zeros_like(flat_k)
        for p in range(ctx):
            flat_k[p] = t["kc"][t["pt"][r, p // P], p % P]
            flat_v[p] = t["vc"][t["pt"][r, p // P], p % P]
        flat_k[ctx:] = t["kn"][c0:c1]
        flat_v[ctx:] = t["vn"][c0:c1]
        nrow = c1 - c0
        mask = np.arange(ctx + nrow)[None, :] <= (ctx + np.arange(nrow))[:, None]
        for i in range(nrow):
            o_i, l_i = [], []
            for h in range(Hq):
                s = scale * flat_k[:, h // G] @ t["q"][c0 + i, h]
                s = np.where(mask[i], s, -np.inf)
                o_i.append(softmax(s) @ flat_v[:, h // G])
                l_i.append(logsumexp(s))
            outs.append(o_i)
            lses.append(l_i)
    return np.array(outs), np.array(lses)


def test_attention_matches_dense_masked_form():
    rng = np.random.default_rng(3)
    t = _toy_gqa(rng, B=3, ctx=(5, 0, 9), n=(3, 2, 4))
    o, lse = O.verify_attention_gqa(t["q"], t["kn"], t["vn"], t["kc"], t["vc"], t["pt"], t["ctx"],
                                    t["cu"], 4, 2, 0.3)
    o2, lse2 = _dense_masked_reference(t, 4, 2, 0.3)
    assert np.allclose(o, o2, atol=1e-12) and np.allclose(lse, lse2, atol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(4)
    t = _toy_gqa(rng, B=2, ctx=(0, 6), n=(2, 3))
    o, lse = O.verify_attention_gqa(t["q"], t["kn"], t["vn"], t["kc"], t["vc"], t["pt"], t["ctx"],
                                    t["cu"], 4, 2, 0.5)
    # empty context, first block row: attends to itself only
    for h in range(4):
        assert np.allclose(o[0, h], t["vn"][0, h // 2])
        assert math.isclose(lse[0, h], 0.5 * t["kn"][0, h // 2] @ t["q"][0, h], rel_tol=1e-12)
    # constant keys -> uniform average of the visible values, lse = s + log(n)
    t2 = dict(t)
    t2["kc"] = np.ones_like(t["kc"])
    t2["kn"] = np.ones_like(t["kn"])
    o, lse = O.verify_attention_gqa(t2["q"], t2["kn"], t2["vn"], t2["kc"], t2["vc"], t2["pt"],
                                    t2["ctx"], t2["cu"], 4, 2, 0.5)
    r, i = 1, 1
    row = t["cu"][r] + i
    vis_v = [t["vc"][t["pt"][r, p // 4], p % 4] for p in range(6)] + [t["vn"][t["cu"][r] + k]
                                                                     for k in range(i + 1)]
    for h in range(4):
        mean = np.mean([v[h // 2] for v in vis_v], axis=0)
        assert np.allclose(o[row, h], mean)
        assert math.isclose(lse[row, h], 0.5 * t["q"][row, h].sum() + math.log(8), rel_tol=1e-12)


def test_attention_page_permutation_and_causality():
    rng = np.random.default_rng(6)
    t = _toy_gqa(rng, B=2, ctx=(7, 3), n=(3, 3))
    base = O.verify_attention_gqa(t["q"], t["kn"], t["vn"], t["kc"], t["vc"], t["pt"], t["ctx"],
                                  t["cu"], 4, 2, 0.4)
    # relabel physical pages: same result
    n_pages = t["kc"].shape[0]
    perm = rng.permutation(n_pages)
    inv = np.argsort(perm)
    kc2, vc2 = t["kc"][perm], t["vc"][perm]
    pt2 = np.where(t["pt"] >= 0, inv[np.maximum(t["pt"], 0)], -1)
    o2 = O.verify_attention_gqa(t["q"], t["kn"], t["vn"], kc2, vc2, pt2, t["ctx"], t["cu"], 4, 2, 0.4)
    assert np.allclose(base[0], o2[0]) and np.allclose(base[1], o2[1])
    # changing block row 2 of request 0 leaves rows 0, 1 untouched
    kn3 = t["kn"].copy()
    kn3[2] += 5.0
    o3 = O.verify_attention_gqa(t["q"], kn3, t["vn"], t["kc"], t["vc"], t["pt"], t["ctx"], t["cu"],
                                4, 2, 0.4)
    assert np.allclose(o3[0][:2], base[0][:2]) and not np.allclose(o3[0][2], base[0][2])


def test_attention_group_to_kv_head_mapping():
    rng = np.random.default_rng(8)
    t = _toy_gqa(rng, B=1, Hq=4, Hkv=2, ctx=(4,), n=(1,))
    t["kc"][:] = 0.0
    t["kn"][:] = 0.0
    page0 = t["pt"][0, 0]
    t["kc"][page0, 2, 1, :] = 40.0           # a dominant key, only on KV head 1, position 2
    t["q"][:] = 1.0
    o, _ = O.verify_attention_gqa(t["q"], t["kn"], t["vn"], t["kc"], t["vc"], t["pt"], t["ctx"],
                                  t["cu"], 4, 2, 1.0)
    # query heads 2, 3 (group of KV head 1) copy that value; heads 0, 1 average uniformly
    assert np.allclose(o[0, 2], t["vc"][page0, 2, 1]) and np.allclose(o[0, 3], t["vc"][page0, 2, 1])
    assert not np.allclose(o[0, 0], t["vc"][page0, 2, 0])


def test_mla_is_shared_latent_mqa():
    rng = np.random.default_rng(9)
    P, Dqk, Dv, H = 4, 12, 8, 3
    ctx, n = (6, 2), (2, 3)
    n_pages = 5
    lc = rng.normal(size=(n_pages, P, Dqk))
    pt = np.array([[3, 1, -1], [4, -1, -1]])
    cu = np.array([0, 2, 5])
    q = rng.normal(size=(5, H, Dqk))
    ln = rng.normal(size=(5, Dqk))
    o, lse = O.verify_attention_mla(q, ln, lc, pt, np.array(ctx), cu, Dv, 0.25)
    # the same computation as GQA with one KV head whose K is the latent and V its first Dv dims
    o2, lse2 = O.verify_attention_gqa(q, ln[:, None, :], ln[:, None, :Dv], lc[:, :, None, :],
                                      lc[:, :, None, :Dv], pt, np.array(ctx), cu, H, 1, 0.25)
    assert np.allclose(o, o2) and np.allclose(lse, lse2)


# ---------------------------------------------------------------- acceptance

def _rows_for(p_pos, cu, B):
    """Lay per-position target rows (B, gamma+1, V) out as packed rows."""
    V = p_pos.shape[-1]
    out = np.zeros((int(cu[-1]), V), np.float32)
    for r in range(B):
        n = cu[r + 1] - cu[r]
        out[cu[r]:cu[r + 1]] = p_pos[r, :n]
    return out


def _three_mode_setup(accept_first=4, gamma=6, V=8, seed=0):
    """Target accepts exactly the first ``accept_first`` drafts: p_t(d_j) >= p_d(d_j)
    for j <= accept_first (always accepted), p_t(d_j) = 0 at the next one."""
    rng = np.random.default_rng(seed)
    p_t = rng.dirichlet(np.ones(V), size=(1, gamma + 1))
    p_d = 0.5 * rng.dirichlet(np.ones(V), size=(1, gamma)) + 0.5 / V
    d = np.zeros((1, gamma), np.int32)
    for j in range(gamma):
        x = int(np.argmax(p_d[0, j]))
        d[0, j] = x
        if j < accept_first:
            p_t[0, j] = 0.3 * p_t[0, j]
            p_t[0, j, x] += 0.7
        elif j == accept_first:
            p_t[0, j, x] = 0.0
            p_t[0, j] /= p_t[0, j].sum()
    p_t, p_d = p_t.astype(np.float32), p_d.astype(np.float32)
    for j in range(min(accept_first, gamma)):
        assert p_t[0, j, d[0, j]] >= p_d[0, j, d[0, j]]
    u = np.full((1, gamma), 0.999, np.float32)
    e = rng.exponential(size=(1, V)).astype(np.float32) + np.float32(1e-3)
    return p_t, p_d, d, u, e


def test_three_mode_example_from_page():
    g = _gold("three_mode_example.json")
    gamma, w, k = g["gamma"], g["window"], g["target_accepts_first"]
    p_t, p_d, d, u, e = _three_mode_setup(k, gamma)
    res = {}
    for name, mode in (("compact", O.COMPACT), ("static", O.STATIC), ("cap_accept", O.CAP_ACCEPT)):
        win = np.array([gamma if mode == O.STATIC else w], np.int32)
        n = gamma + 1 if mode != O.COMPACT else w + 1
        cu = np.array([0, n])
        a = O.accept(_rows_for(p_t, cu, 1), p_d, d, u, e, win, cu, mode, gamma)
        res[name] = a
        assert a.accept_len[0] == g["expect"][name]["accept_len"]
        assert a.cap_len[0] == g["expect"][name]["cap_len"]
    bonus = int(np.argmax((p_t[0, w] / e[0]).astype(np.float32)))
    assert res["compact"].out_tok[0] == bonus
    assert res["cap_accept"].out_tok[0] == res["compact"].out_tok[0]
    resid = np.maximum(0, p_t[0, k] - p_d[0, k]).astype(np.float32)
    assert res["static"].out_tok[0] == int(np.argmax((resid / e[0]).astype(np.float32)))


def test_prefix_semantics_from_page():
    g = _gold("prefix_example.json")
    gamma = g["gamma"]
    p_t, p_d, d, u, e = _three_mode_setup(g["reject_at"] - 1, gamma, seed=3)
    # make the drafts after the rejection individually acceptable
    for j in range(g["reject_at"], gamma):
        p_t[0, j, d[0, j]] = 1.0
    cu = np.array([0, gamma + 1])
    a = O.accept(_rows_for(p_t, cu, 1), p_d, d, u, e, np.array([gamma], np.int32), cu,
                 O.STATIC, gamma)
    assert a.accept_len[0] == g["accept_len"]


def test_identical_and_disjoint_distributions():
    rng = np.random.default_rng(12)
    V, gamma = 16, 4
    p = rng.dirichlet(np.ones(V), size=(1, gamma + 1)).astype(np.float32)
    d = np.array([[int(np.argmax(p[0, j])) for j in range(gamma)]], np.int32)
    u = rng.uniform(0.01, 0.99, size=(1, gamma)).astype(np.float32)
    e = rng.exponential(size=(1, V)).astype(np.float32) + np.float32(1e-3)
    cu = np.array([0, gamma + 1])
    a = O.accept(_rows_for(p, cu, 1), p[:, :gamma].copy(), d, u, e, np.array([gamma], np.int32),
                 cu, O.COMPACT, gamma)
    assert a.accept_len[0] == gamma and np.allclose(a.cstar, 1.0, atol=1e-6)
    # disjoint supports: c* = 0 and the first draft is rejected
    pt = np.zeros((1, gamma + 1, V), np.float32)
    pt[..., : V // 2] = 2.0 / V
    pd = np.zeros((1, gamma, V), np.float32)
    pd[..., V // 2:] = 2.0 / V
    d2 = np.full((1, gamma), V - 1, np.int32)
    a2 = O.accept(_rows_for(pt, cu, 1), pd, d2, u, e, np.array([gamma], np.int32), cu,
                  O.COMPACT, gamma)
    assert a2.accept_len[0] == 0 and np.allclose(a2.cstar, 0.0, atol=1e-7)
    assert a2.out_tok[0] < V // 2           # the correction comes from the target's support


@pytest.mark.parametrize("mode", [O.COMPACT, O.STATIC, O.CAP_ACCEPT])
def test_cstar_positions_and_hand_values(mode):
    """c* (reading A13) exists for the draft positions whose target row was verified:
    j = 1..min(w + 1, gamma) in compact mode, 1..gamma in static and cap-accept; the
    others are NaN.  Values by hand: identical rows give 1; p_t = (1/2, 1/2, 0, 0)
    against a uniform draft gives 1 - (1/4 + 1/4 + 1/4 + 1/4) / 2 = 1/2; a target row
    (1, 0, 0, 0) against (0, 1/2, 1/2, 0) gives 0."""
    gamma, V, w = 4, 4, 1
    q = np.full(V, 0.25, np.float32)
    half = np.array([0.5, 0.5, 0.0, 0.0], np.float32)
    one = np.array([1.0, 0.0, 0.0, 0.0], np.float32)
    mid = np.array([0.0, 0.5, 0.5, 0.0], np.float32)
    p_d = np.stack([q, q, mid, q])[None]                  # draft rows j = 1..4
    p_t = np.stack([q, half, one, q, q])[None]            # target rows 0..4
    d = np.zeros((1, gamma), np.int32)                    # the target keeps mass on 0
    u = np.full((1, gamma), 0.5, np.float32)
    e = np.ones((1, V), np.float32)
    win = np.array([gamma if mode == O.STATIC else w], np.int32)
    n = w + 1 if mode == O.COMPACT else gamma + 1
    cu = np.array([0, n])
    a = O.accept(_rows_for(p_t, cu, 1), p_d, d, u, e, win, cu, mode, gamma)
    c = a.cstar[0]
    assert c[0] == 1.0 and c[1] == 0.5
    if mode == O.COMPACT:
        assert np.isnan(c[2]) and np.isnan(c[3])
    else:
        assert c[2] == 0.0 and c[3] == 1.0


def test_race_argmax_lowest_index_on_ties():
    w = np.array([0.1, 0.4, 0.2, 0.4], np.float32)
    e = np.ones(4, np.float32)
    assert O._race_argmax(w, e)[0] == 1


@pytest.mark.parametrize("window", [0, 1, 2])
def test_acceptance_preserves_target_distribution(window):
    """Textbook speculative sampling: the first committed token is distributed
    exactly as the target at position 1, whatever the draft distribution."""
    rng = np.random.default_rng(20 + window)
    V, gamma, N = 6, 2, 30000
    p_t1 = rng.dirichlet(np.ones(V) * 0.8).astype(np.float32)
    p_d1 = rng.dirichlet(np.ones(V) * 0.8).astype(np.float32)
    p_t = np.tile(p_t1, (N, gamma + 1, 1))
    p_d = np.tile(p_d1, (N, gamma, 1))
    d = np.stack([rng.choice(V, size=N, p=p_d1 / p_d1.sum()) for _ in range(gamma)], 1).astype(np.int32)
    u = ((rng.integers(0, 1 << 24, size=(N, gamma)) + 0.5) * 2.0 ** -24).astype(np.float32)
    e = (-np.log((rng.integers(0, 1 << 24, size=(N, V)) + 0.5) * 2.0 ** -24)).astype(np.float32)
    win = np.full(N, window, np.int32)
    cu = np.arange(N + 1) * (window + 1)
    rows = np.repeat(p_t1[None], int(cu[-1]), 0)
    a = O.accept(rows, p_d, d, u, e, win, cu, O.COMPACT, gamma)
    first = np.where(a.accept_len > 0, d[:, 0], a.out_tok)
    counts = np.bincount(first, minlength=V)
    expected = p_t1.astype(np.float64) / p_t1.sum() * N
    chi2 = ((counts - expected) ** 2 / expected).sum()
    assert stats.chi2.sf(chi2, V - 1) > 1e-4


# ---------------------------------------------------------------- compaction

def test_compact_hand_worked_example():
    g = _gold("compact_example.json")
    P = g["page_size"]
    B = 3
    L = np.array(g["accept_len"], np.int32)
    cu = np.concatenate([[0], np.cumsum(L + 1)]).astype(np.int32)
    M = int(cu[-1])
    kn = np.arange(M, dtype=np.float32).reshape(M, 1, 1) + 100.0
    kc = np.zeros((8, P, 1, 1), np.float32)
    draft = np.arange(B * 5).reshape(B, 5).astype(np.int32)
    tok = np.array([70, 71, 72], np.int32)
    c = O.compact(kn, kn, cu, L, tok, draft, P, np.array(g["page_table"]), np.array(g["ctx_len"]),
                  np.array([1, 2, 3]), np.array(g["free_pages"]), g["free_top"], kc, kc.copy())
    assert c.page_table.tolist() == g["expect_page_table"]
    assert c.ctx_len.tolist() == g["expect_ctx_len"] and c.free_top == g["expect_free_top"]
    for r, slots in g["expect_slots"].items():
        r = int(r)
        for i, (page, off) in enumerate(slots):
            assert c.k_cache[page, off, 0, 0] == 100.0 + cu[r] + i
    assert c.anchor.tolist() == [70, 71, 72]
    assert c.committed[2].tolist() == [10, 11, 12, 13, 72, -1]
    assert c.n_committed.tolist() == [3, 1, 5]


@pytest.mark.parametrize("seed", range(6))
def test_compact_invariants_on_random_states(seed):
    """Commit invariants on random states (page sizes 1..16, contexts on and off page
    boundaries, windows 0..gamma): the committed counts sum to sum(L + 1) and hold
    d_1..d_L then the token; old page-table entries are unchanged; the new entries are
    the top sum(new pages) entries of the free stack, taken in request order (so each
    page once, none already held); free_top drops by their number; ctx grows by L + 1
    and the anchor is the token; every kept row lands at its position through the new
    table, and no other cache slot changes."""
    rng = np.random.default_rng(100 + seed)
    B, gamma = int(rng.integers(1, 13)), int(rng.integers(2, 9))
    P = int(rng.choice([1, 2, 4, 16]))
    max_pages = (6 * P + gamma + 4) // P + 2
    ctx = rng.integers(0, 5 * P + 4, B).astype(np.int32)
    L = rng.integers(0, gamma + 1, B).astype(np.int32)
    have = (ctx + P - 1) // P
    n_pages = int(have.sum()) + B * max_pages + 3
    perm = rng.permutation(n_pages).astype(np.int32)
    pt = np.full((B, max_pages), -1, np.int32)
    o = 0
    for r in range(B):
        pt[r, :have[r]] = perm[o:o + have[r]]
        o += int(have[r])
    free = perm[o:].copy()
    top = len(free) - int(rng.integers(0, 3))  # entries above top are not free
    cu = np.concatenate([[0], np.cumsum(L + 1 + rng.integers(0, 3, B))]).astype(np.int32)
    M = int(cu[-1])
    kn = (np.arange(M, dtype=np.float32) + 1000.0).reshape(M, 1, 1)
    vn = -kn
    kc = -(np.arange(n_pages * P, dtype=np.float32) + 1.0).reshape(n_pages, P, 1, 1)
    vc = kc * 3.0
    draft = rng.integers(0, 50000, (B, gamma)).astype(np.int32)
    tok = rng.integers(0, 50000, B).astype(np.int32)
    anchor = rng.integers(0, 50000, B).astype(np.int32)
    c = O.compact(kn, vn, cu, L, tok, draft, P, pt, ctx, anchor, free, top, kc, vc)
    keep = L + 1
    nn = (ctx + keep + P - 1) // P - have
    assert int(c.n_committed.sum()) == int(keep.sum())
    for r in range(B):
        assert c.committed[r, :L[r]].tolist() == draft[r, :L[r]].tolist()
        assert c.committed[r, L[r]] == tok[r] and (c.committed[r, L[r] + 1:] == -1).all()
    assert (c.ctx_len == ctx + keep).all() and (c.anchor == tok).all()
    assert c.free_top == top - int(nn.sum())
    held = set(int(x) for x in pt[pt >= 0])
    taken = []
    for r in range(B):
        assert (c.page_table[r, :have[r]] == pt[r, :have[r]]).all()        # old entries
        assert (c.page_table[r, have[r] + nn[r]:] == -1).all()
        taken += c.page_table[r, have[r]:have[r] + nn[r]].tolist()
    assert taken == free[top - int(nn.sum()):top][::-1].tolist()          # stack order
    assert len(set(taken)) == len(taken) and not (set(taken) & held)
    changed = np.zeros(kc.shape[:2], bool)
    for r in range(B):
        for i in range(int(keep[r])):
            pos = int(ctx[r]) + i
            page = int(c.page_table[r, pos // P])
            assert c.k_cache[page, pos % P, 0, 0] == kn[cu[r] + i, 0, 0]
            assert c.v_cache[page, pos % P, 0, 0] == vn[cu[r] + i, 0, 0]
            changed[page, pos % P] = True
    assert (c.k_cache[~changed] == kc[~changed]).all()
    assert (c.v_cache[~changed] == vc[~changed]).all()


def test_compact_no_space_raises():
    kn = np.zeros((2, 1, 1), np.float32)
    with pytest.raises(O.NoSpace):
        O.compact(kn, kn, np.array([0, 2]), np.array([1]), np.array([0]), np.zeros((1, 3), np.int32),
                  2, np.array([[0, -1]]), np.array([2]), np.array([0]), np.array([], np.int32), 0,
                  np.zeros((2, 2, 1, 1)), np.zeros((2, 2, 1, 1)))


# ---------------------------------------------------------------- confidence sigmoid

def _ulps(a, b):
    a = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    b = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    return np.abs(a - b)


def test_confidence_sigmoid_hand_values():
    """sigma(0) = 1/2, sigma(ln 3) = 3/4, sigma(-ln 3) = 1/4: the fp32 rounding of
    ln 3 moves sigma by about 4e-9, under half an ulp of 3/4 and of 1/4, so all
    three are exact; a sign flip or a dropped term gives 1/4 for 3/4."""
    z = np.array([[0.0, math.log(3.0), -math.log(3.0)]], np.float32)
    c = O.confidence(z, True)
    assert c[0].tolist() == [0.5, 0.75, 0.25]
    # is_logit = 0 passes the confidence through unchanged
    x = np.array([[0.3, 0.9]], np.float32)
    assert np.array_equal(O.confidence(x, False), x)


def test_confidence_sigmoid_matches_scipy_expit():
    from scipy.special import expit
    z = np.linspace(-30, 30, 2001, dtype=np.float32)[None, :]
    c = O.confidence(z, True)
    ref = expit(z.astype(np.float64)).astype(np.float32)
    assert np.all(_ulps(c, ref) <= 1)
    assert np.all(np.diff(c[0]) >= 0) and c[0, 0] < 1e-12 and c[0, -1] == 1.0


# ---------------------------------------------------------------- race rule (reading A11)

def test_race_zero_weight_never_wins_even_with_zero_noise():
    """w / e with w = 0 and e = 0 is NaN; the entry must still lose to any positive
    weight (log 0 = -inf in the Gumbel form)."""
    w = np.array([0.0, 0.25, 0.0, 0.1], np.float32)
    e = np.array([0.0, 1.0, 0.0, 5.0], np.float32)
    idx, key, live = O._race_argmax(w, e)
    assert (idx, live) == (1, True) and key == 0.25
    # a NaN noise entry on a positive weight is not a winner either
    e2 = np.array([1.0, np.nan, 1.0, 5.0], np.float32)
    assert O._race_argmax(w, e2)[0] == 3


def test_race_all_zero_weights_give_index_zero_and_no_live_entry():
    idx, key, live = O._race_argmax(np.zeros(5, np.float32), np.ones(5, np.float32))
    assert (idx, live) == (0, False) and key == float("-inf")


def test_race_infinite_keys_tie_to_lowest_index():
    """e = 0 on positive weights gives +inf keys: the lowest such index wins."""
    w = np.array([0.5, 0.0, 0.2, 0.3], np.float32)
    e = np.array([1.0, 0.0, 0.0, 0.0], np.float32)
    assert O._race_argmax(w, e)[0] == 2


def test_race_positive_weight_with_underflowing_key_beats_zero_weights():
    """A positive weight whose quotient rounds to 0 is still a live entry: it wins
    against zero weights (which are -inf), lowest index among equal keys."""
    w = np.array([0.0, 1e-44, 0.0], np.float32)
    e = np.array([1.0, 1e30, 1.0], np.float32)
    idx, key, live = O._race_argmax(w, e)
    assert (idx, key, live) == (1, 0.0, True)


def test_correction_fallback_only_without_any_positive_residual():
    """Reading A12: the p_t fallback is taken iff max(0, p_t - p_d) has no positive
    entry; a residual whose only positive entry gives a zero key is still raced."""
    V, gamma = 4, 1
    pt = np.array([[0.25, 0.25, 0.25, 0.25], [0.25, 0.25, 0.25, 0.25]], np.float32)
    d = np.array([[0]], np.int32)
    u = np.array([[0.99]], np.float32)
    e = np.array([[1.0, 1.0, 1e30, 1.0]], np.float32)
    cu = np.array([0, 2])
    # rejected draft, residual zero everywhere -> fallback to p_t
    pd0 = np.array([[[0.5, 0.25, 0.25, 0.25]]], np.float32)
    a = O.accept(pt, pd0, d, u, e, np.array([1], np.int32), cu, O.COMPACT, gamma)
    assert a.accept_len[0] == 0 and a.residual_fallback[0] and a.out_tok[0] == 0
    # one tiny positive residual entry at index 2 whose key underflows to 0 -> no fallback
    pd1 = pd0.copy()
    pd1[0, 0, 2] = np.nextafter(np.float32(0.25), np.float32(0))
    a1 = O.accept(pt, pd1, d, u, e, np.array([1], np.int32), cu, O.COMPACT, gamma)
    assert not a1.residual_fallback[0] and a1.out_tok[0] == 2


# ---------------------------------------------------------------- input generator

def test_generator_uniforms_are_exact_and_open():
    """The seeded uniforms are odd multiples of 2^-24 (exact fp32, never 0 or 1) and
    the exponential noise -log u is finite and strictly positive."""
    import torch
    import workloads as W
    wl = W.WORKLOADS["tiny"].replace(B=64, vocab=4096)
    inp = W.make_inputs(wl, 9)
    for u in (inp["uniforms"],):
        k = u.to(torch.float64) * 2.0 ** 24
        assert torch.all(k == torch.round(k)) and torch.all(torch.remainder(k, 2) == 1)
        assert float(u.min()) > 0.0 and float(u.max()) < 1.0
    e = inp["exp_noise"]
    assert torch.all(torch.isfinite(e)) and float(e.min()) > 0.0


# ---------------------------------------------------------------- calibration tooling

def test_calib_samples_label_rule():
    """Verified positions only; label 1 iff the accepted prefix reaches the position."""
    a = np.array([[0.9, 0.8, 0.5], [0.7, 0.6, 0.2]], np.float32)
    ah = a * np.float32(0.5)
    s = O.calib_samples(a, ah, np.array([2, 0], np.int32), np.array([1, 0], np.int32),
                        O.COMPACT, 3)
    assert [[y for (_, _, y) in pos] for pos in s] == [[1], [0], []]
    assert s[0][0][0] == np.float32(0.9) and s[0][0][1] == np.float32(0.45)
    # cap-accept verifies the whole block: every position of every request is labelled
    s2 = O.calib_samples(a, ah, np.array([2, 0], np.int32), np.array([2, 0], np.int32),
                         O.CAP_ACCEPT, 3)
    assert [[y for (_, _, y) in pos] for pos in s2] == [[1, 0], [1, 0], [0, 0]]


def test_ece_hand_example_and_one_bin_identity():
    p = [0.1, 0.45, 0.55, 0.95]
    y = [0, 0, 1, 1]
    samples = [[(np.float32(0.5), np.float32(pi), yi) for pi, yi in zip(p, y)]]
    e, cnt, sp, sy = O.ece(samples, 2)
    # bin 0: p 0.1, 0.45 (sum 0.55), y 0;  bin 1: p 0.55, 0.95 (sum 1.5), y 2
    assert cnt.tolist() == [2, 2] and sy.tolist() == [0.0, 2.0]
    assert abs(e - (0.55 + 0.5) / 4) < 1e-7
    # one bin: |mean(y) - mean(p)|
    e1, _, _, _ = O.ece(samples, 1)
    assert abs(e1 - abs(2 - sum(float(np.float32(x)) for x in p)) / 4) < 1e-12
    # bin edges: p = 1 falls in the last bin, p = 0.5 in the upper of two
    e2, c2, _, _ = O.ece([[(0.5, np.float32(1.0), 1), (0.5, np.float32(0.5), 1)]], 2)
    assert c2.tolist() == [0, 2] and abs(e2 - 0.25) < 1e-12
    assert O.ece([[]], 10)[0] == 0.0


def test_ece_of_calibrated_predictions_is_small():
    rng = np.random.default_rng(31)
    p = rng.uniform(0, 1, 200_000).astype(np.float32)
    y = (rng.uniform(0, 1, p.size) < p).astype(int)
    e, _, _, _ = O.ece([[(0.5, pi, yi) for pi, yi in zip(p, y)]], 10)
    assert e < 0.01
    # a miscalibrated predictor (p^2 against labels drawn with p) has a clearly larger ECE
    e_bad, _, _, _ = O.ece([[(0.5, np.float32(pi * pi), yi) for pi, yi in zip(p, y)]], 10)
    assert e_bad > 0.1


def _logit_samples(z, y):
    a = (1.0 / (1.0 + np.exp(-z))).astype(np.float32)
    return [(ai, ai, int(yi)) for ai, yi in zip(a, y)]


def test_sts_fit_recovers_the_temperature_and_the_optimum():
    """Labels drawn with probability sigmoid(z / T_true): the refit is the exact
    minimiser of the binary cross-entropy (checked against scipy's bounded scalar
    minimiser) and lies within a few standard errors of T_true."""
    from scipy.optimize import minimize_scalar
    rng = np.random.default_rng(32)
    T_true = 1.7
    z = rng.normal(0.0, 2.5, 20_000)
    y = (rng.uniform(0, 1, z.size) < 1.0 / (1.0 + np.exp(-z / T_true))).astype(int)
    samples = _logit_samples(z, y)
    T = float(O.sts_fit(samples, 60))
    za = np.array([float(np.log(a) - np.log1p(-a)) for (a, _, _) in samples])

    def nll(lb):
        t = np.exp(lb) * za
        return float(np.sum(np.logaddexp(0.0, t) - y * t))
    res = minimize_scalar(nll, bounds=(-3, 3), method="bounded", options={"xatol": 1e-12})
    assert abs(T - float(np.exp(-res.x))) < 1e-5 * T
    assert abs(T - T_true) < 0.1 * T_true


def test_sts_fit_degenerate_cases():
    # no sample, or only a = 1 (infinite logit): the identity temperature
    assert O.sts_fit([], 40) == np.float32(1.0)
    assert O.sts_fit([(np.float32(1.0), np.float32(1.0), 1)], 40) == np.float32(1.0)
    # every positive logit accepted and every negative one rejected: the sharpest
    # temperature the range allows (beta clamped at 64)
    s = [(np.float32(0.8), np.float32(0.8), 1), (np.float32(0.3), np.float32(0.3), 0)]
    T = float(O.sts_fit(s, 60))
    assert abs(T - 1.0 / 64) < 1e-6


# ---------------------------------------------------------------- Markov-head draft sampling

def test_markov_without_bias_is_the_backbone_softmax():
    """W2 = 0: the Markov head adds nothing, so p_k = softmax(U_k) at every position
    whatever the previous tokens (checked against scipy's softmax)."""
    from scipy.special import softmax
    rng = np.random.default_rng(40)
    B, gamma, V, r = 3, 4, 37, 8
    U = rng.normal(0, 3, (B, gamma, V)).astype(np.float32)
    W1 = rng.normal(0, 1, (V, r))
    W2 = np.zeros((r, V))
    e = rng.exponential(size=(B, gamma, V)).astype(np.float32)
    _, P, _ = O.markov_draft(U, W1, W2, np.array([0, 5, 36]), e)
    np.testing.assert_allclose(P, softmax(U.astype(np.float64), axis=-1), rtol=1e-12, atol=0)


def test_markov_chain_follows_the_previous_token():
    """A dominant transition bias B(x, v) = 50 [v == x + 1 mod V] (W1 = 50 I, W2 the
    shift) with flat backbone logits: each position takes the token after the previous
    one, starting from the anchor -- a bias read from the anchor at every position,
    or from any other position, gives another chain."""
    V = 8
    W1 = 50.0 * np.eye(V)
    W2 = np.roll(np.eye(V), 1, axis=1)          # W2[i, (i + 1) % V] = 1
    B, gamma = 3, 6
    U = np.zeros((B, gamma, V), np.float32)
    rng = np.random.default_rng(41)
    e = rng.uniform(0.5, 2.0, (B, gamma, V)).astype(np.float32)
    anchor = np.array([0, 3, 7])
    tok, P, _ = O.markov_draft(U, W1, W2, anchor, e)
    for b in range(B):
        assert tok[b].tolist() == [(anchor[b] + k + 1) % V for k in range(gamma)]
    assert np.all(P.max(-1) >= 1 - 1e-15)


def test_markov_race_is_the_gumbel_max():
    """The exponential race argmax p / e is the Gumbel-max argmax log p + G with
    G = -log e, by brute force over every entry, and equal keys go to the lowest index."""
    rng = np.random.default_rng(42)
    B, gamma, V, r = 4, 3, 23, 5
    U = rng.normal(0, 2, (B, gamma, V)).astype(np.float32)
    W1 = rng.normal(0, 0.5, (V, r))
    W2 = rng.normal(0, 0.5, (r, V))
    e = rng.exponential(size=(B, gamma, V)).astype(np.float32)
    tok, P, _ = O.markov_draft(U, W1, W2, rng.integers(0, V, B), e)
    for b in range(B):
        for k in range(gamma):
            gumbel = np.log(P[b, k]) - np.log(e[b, k].astype(np.float64))
            assert tok[b, k] == int(np.argmax(gumbel))
    # ties: flat logits, no bias, equal noise -> every key equal -> index 0
    tok, _, _ = O.markov_draft(np.zeros((1, 2, 9), np.float32), np.zeros((9, 2)),
                               np.zeros((2, 9)), np.array([4]), np.ones((1, 2, 9), np.float32))
    assert tok.tolist() == [[0, 0]]


def test_markov_conditioning_on_given_tokens():
    """With tokens_given, position k is the one-step draw after tokens_given[:, k-1]:
    the same p as a one-position block whose anchor is that token."""
    rng = np.random.default_rng(43)
    B, gamma, V, r = 2, 4, 19, 6
    U = rng.normal(0, 2, (B, gamma, V)).astype(np.float32)
    W1 = rng.normal(0, 1, (V, r))
    W2 = rng.normal(0, 1, (r, V))
    e = rng.exponential(size=(B, gamma, V)).astype(np.float32)
    given = rng.integers(0, V, (B, gamma))
    _, P, _ = O.markov_draft(U, W1, W2, np.array([1, 2]), e, tokens_given=given)
    for k in range(1, gamma):
        _, P1, _ = O.markov_draft(U[:, k:k + 1], W1, W2, given[:, k - 1], e[:, k:k + 1])
        np.testing.assert_allclose(P[:, k], P1[:, 0], rtol=0, atol=0)


# ------------------------------------------------------------------ block-accept estimate

def _estimate_case(rng, B=64, gamma=6, V=16):
    """Per-position target rows for positions 1..gamma+1 (the same rows in every mode,
    reading A18), drafter rows, drafts drawn from them, uniforms, windows 0..gamma;
    the target leans towards the drafter by a per-request amount so that accepted
    prefixes of every length occur."""
    p_d = rng.dirichlet(np.ones(V) * 0.5, size=(B, gamma)).astype(np.float32)
    mix = rng.uniform(0.0, 1.0, size=(B, 1, 1))
    mix[:2] = 1.0   # p_t = p_d: every draft is accepted (u < 1)
    rnd = rng.dirichlet(np.ones(V) * 0.5, size=(B, gamma + 1))
    pd_ext = np.concatenate([p_d, p_d[:, -1:]], axis=1)
    p_t = (mix * pd_ext + (1 - mix) * rnd).astype(np.float32)
    def draw(row):
        q = row.astype(np.float64)
        return rng.choice(V, p=q / q.sum())
    d = np.array([[draw(p_d[r, j]) for j in range(gamma)] for r in range(B)], np.int32)
    u = rng.uniform(1e-6, 1.0, size=(B, gamma)).astype(np.float32)
    e = rng.exponential(size=(B, V)).astype(np.float32) + np.float32(1e-3)
    win = rng.integers(0, gamma + 1, size=B).astype(np.int32)
    win[0], win[1] = gamma, gamma // 2   # a whole-block window; an open interval
    return p_t, p_d, d, u, e, win


@pytest.mark.parametrize("seed", range(4))
def test_block_accept_estimate_brackets_the_full_block_cap(seed):
    """The interval from a compact run contains the cap a cap-accept run on the same
    inputs sees (the definition of the censored quantity), and is exact wherever the
    compact run holds the deciding test: a rejection inside the window, the whole
    block as window, or a rejection at position w + 1 (the bonus row)."""
    rng = np.random.default_rng(100 + seed)
    gamma = 6
    p_t, p_d, d, u, e, win = _estimate_case(rng, gamma=gamma)
    B = len(win)
    cu_c = np.concatenate([[0], np.cumsum(1 + win)])
    a_c = O.accept(_rows_for(p_t, cu_c, B), p_d, d, u, e, win, cu_c, O.COMPACT, gamma)
    full = np.full(B, gamma, np.int32)
    cu_f = np.concatenate([[0], np.cumsum(1 + full)])
    a_f = O.accept(_rows_for(p_t, cu_f, B), p_d, d, u, e, win, cu_f, O.CAP_ACCEPT, gamma)
    lo, hi = O.block_accept_estimate(_rows_for(p_t, cu_c, B), p_d, d, u, win, cu_c,
                                     a_c.accept_len, a_c.cap_len, O.COMPACT, gamma)
    cap = a_f.cap_len
    assert np.all(lo <= cap) and np.all(cap <= hi)
    for r in range(B):
        w, L = int(win[r]), int(a_c.accept_len[r])
        if L < w or w == gamma or cap[r] == w:
            assert lo[r] == hi[r] == cap[r], r
        else:   # the test at w + 1 accepted: only the lower end is known
            assert (lo[r], hi[r]) == (w + 1, gamma) and cap[r] >= w + 1, r
    # every kind of case occurs
    kinds = {("in" if a_c.accept_len[r] < win[r] else "full" if win[r] == gamma else
              "w+1 rejects" if lo[r] == hi[r] else "open") for r in range(B)}
    assert kinds == {"in", "full", "w+1 rejects", "open"}
    # the other modes report the cap they verified
    for mode in (O.STATIC, O.CAP_ACCEPT):
        lo2, hi2 = O.block_accept_estimate(_rows_for(p_t, cu_f, B), p_d, d, u, full, cu_f,
                                           a_f.accept_len, a_f.cap_len, mode, gamma)
        assert np.array_equal(lo2, a_f.cap_len) and np.array_equal(hi2, a_f.cap_len)


@pytest.mark.parametrize("accept_first", [2, 3, 4])
def test_block_accept_estimate_on_the_page_example(accept_first):
    """The three-mode example of [lesson] "Confidence scheduler 与 verify 模式" (block 6,
    window 3) with the target accepting the first k drafts: a rejection inside the
    window (k = 2) gives 2; the rejection right after the window (k = 3) is seen in the
    bonus row and gives 3; the page's own case (k = 4, the cap that cap-accept exposes)
    gives the interval [4, 6], which holds the cap-accept run's cap."""
    g = _gold("three_mode_example.json")
    gamma, w = g["gamma"], g["window"]
    p_t, p_d, d, u, e = _three_mode_setup(accept_first, gamma)
    win = np.array([w], np.int32)
    cu = np.array([0, w + 1])
    a = O.accept(_rows_for(p_t, cu, 1), p_d, d, u, e, win, cu, O.COMPACT, gamma)
    lo, hi = O.block_accept_estimate(_rows_for(p_t, cu, 1), p_d, d, u, win, cu, a.accept_len,
                                     a.cap_len, O.COMPACT, gamma)
    want = {2: (2, 2), 3: (3, 3), 4: (4, gamma)}[accept_first]
    assert (int(lo[0]), int(hi[0])) == want
    if accept_first == g["target_accepts_first"]:
        assert lo[0] <= g["expect"]["cap_accept"]["cap_len"] <= hi[0]

"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the same
seeded inputs.  Integers bit-exact (window decisions the oracle lists as
within 1e-5 relative are reported, not failed); attention max-abs <= 1e-2 and
mean-abs <= 1e-3 against fp64; c* within 1e-5.

lse within 4e-3: the GQA kernel multiplies V by P rounded to bf16 (8 significant
bits: relative error at most 2^-8) and divides by the sum of those same rounded
P, so that the weights applied to V are exactly normalised; its lse = m + log(sum
of rounded P) then differs from the exact one by at most ln(1 + 2^-8) = 3.9e-3
(plus fp32 rounding far below that)."""
import math

import numpy as np
import pytest
import torch

import harness
import workloads as W
from oracle import dspark_oracle as O

pytestmark = pytest.mark.gpu

ATT_MAX, ATT_MEAN, LSE_MAX, CSTAR_TOL = 1e-2, 1e-3, 4e-3, 1e-5
MODES = {"compact": O.COMPACT, "static": O.STATIC, "cap_accept": O.CAP_ACCEPT}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def npy(t):
    if t is None:
        return None
    t = t.detach()
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.cpu().numpy()


def small_np(inp):
    keep = ("conf", "sts_temp", "cost_table", "tiers", "ctx_len", "anchor", "draft_tok",
            "uniforms", "page_table", "free_pages", "free_top")
    return {k: npy(inp[k]) for k in keep}


# ------------------------------------------------------------------ checks

def check_schedule(g, sch, B):
    """Windows bit-exact, except the decisions the oracle lists as within 1e-5
    relative of their margin: those are reported, not failed.  Returns the windows
    the later stages are checked on (the GPU's own when a listed decision went the
    other way, so that every stage is still compared on identical inputs)."""
    ow = sch.windows
    gw = g["windows"].numpy()
    # calibrated survival: identical up to one fp32 ulp (fp64 exp/log of two libraries,
    # each rounded once to fp32)
    ga = g["a_hat"].numpy()
    assert np.all(np.abs(ga.view(np.int32).astype(np.int64) - sch.a_hat.view(np.int32)) <= 1)
    if not sch.listed:
        assert np.array_equal(gw, ow), (gw, ow)
        assert g["M"] == sch.M
        assert math.isclose(g["E"], sch.E, rel_tol=1e-9)
        return ow
    print(f"listed near-margin decisions: {sch.listed}")
    if any(kind == "accept" for (kind, _, _, _) in sch.listed):
        # an accepted candidate within the margin: if it flipped, every later decision
        # moved with it, so only the greedy's shape is checked
        assert g["M"] == B + int(gw.sum())
    else:
        listed_r = {r for (_, r, _, _) in sch.listed}
        other = [r for r in range(B) if r not in listed_r]
        assert np.array_equal(gw[other], ow[other])
    if not np.array_equal(gw, ow):
        print(f"listed decision went the other way: GPU windows {gw.tolist()}")
    return gw


def check_pack(g, pk):
    assert np.array_equal(g["cu_seqlens"].numpy(), pk.cu_seqlens)
    assert g["M_pack"] == pk.M and g["tier"] == pk.tier
    t = pk.tier
    assert np.array_equal(g["row_req"].numpy()[:t], pk.row_req)
    assert np.array_equal(g["row_pos"].numpy()[:t], pk.row_pos)
    assert np.array_equal(g["row_tok"].numpy()[:t], pk.row_tok)


def check_attention(g_out, g_lse, o, lse, rows=None):
    go, gl = g_out, g_lse
    if rows is not None:
        go, gl, o, lse = go[rows], gl[rows], o[rows], lse[rows]
    assert np.all(np.isfinite(go)) and np.all(np.isfinite(gl))
    err = np.abs(go - o)
    assert err.max() <= ATT_MAX and err.mean() <= ATT_MEAN, (err.max(), err.mean())
    assert np.abs(gl - lse).max() <= LSE_MAX, np.abs(gl - lse).max()


def check_accept(g, acc):
    assert np.array_equal(g["accept_len"].numpy(), acc.accept_len)
    assert np.array_equal(g["cap_len"].numpy(), acc.cap_len)
    assert np.array_equal(g["out_tok"].numpy(), acc.out_tok)
    assert np.array_equal(g["fallback"].numpy().astype(bool), acc.residual_fallback)
    cs = g["cstar"].numpy()
    assert np.array_equal(np.isnan(cs), np.isnan(acc.cstar))
    if np.any(~np.isnan(cs)):
        assert np.nanmax(np.abs(cs - acc.cstar)) <= CSTAR_TOL


def oracle_compact_state(inp_np, pk, acc, wl):
    """Integer state after compaction (dummy one-element rows: the cache bytes are
    checked separately, slot by slot)."""
    n_pages = int(np.max(inp_np["page_table"])) + 1 + len(inp_np["free_pages"])
    M = int(pk.cu_seqlens[-1])
    dummy_rows = np.zeros((max(M, 1), 1), np.float32)
    dummy_cache = np.zeros((n_pages, wl.page_size, 1), np.float32)
    return O.compact(dummy_rows, None, pk.cu_seqlens, acc.accept_len, acc.out_tok,
                     inp_np["draft_tok"], wl.page_size, inp_np["page_table"], inp_np["ctx_len"],
                     inp_np["anchor"], inp_np["free_pages"], int(inp_np["free_top"][0]),
                     dummy_cache, None)


def check_compact(g, cm, inp, pk, acc, wl, d_packed):
    assert np.array_equal(g["page_table"].numpy(), cm.page_table)
    assert np.array_equal(g["ctx_len"].numpy(), cm.ctx_len)
    assert np.array_equal(g["anchor"].numpy(), cm.anchor)
    assert g["free_top"] == cm.free_top
    assert np.array_equal(g["committed"].numpy(), cm.committed)
    assert np.array_equal(g["n_committed"].numpy(), cm.n_committed)
    # cache bytes at every newly written slot equal the packed block row
    P = wl.page_size
    ctx0 = npy(inp["ctx_len"])
    slots, rows = [], []
    for r in range(wl.B):
        for i in range(int(acc.accept_len[r]) + 1):
            pos = int(ctx0[r]) + i
            slots.append((int(cm.page_table[r, pos // P]), pos % P))
            rows.append(int(pk.cu_seqlens[r]) + i)
    pages = torch.tensor([s[0] for s in slots], device=g["k_cache"].device)
    offs = torch.tensor([s[1] for s in slots], device=g["k_cache"].device)
    ridx = torch.tensor(rows, device=g["k_cache"].device)
    assert torch.equal(g["k_cache"][pages, offs], d_packed["k_new"][ridx])
    if g.get("v_cache") is not None:
        assert torch.equal(g["v_cache"][pages, offs], d_packed["v_new"][ridx])


def sub_cache(inp, r):
    """Request r's pages relabelled 0..n-1 (attention does not depend on page labels)."""
    P = inp["workload"].page_size
    ctx = int(inp["ctx_len"][r])
    n = (ctx + P - 1) // P
    pages = inp["page_table"][r, :n].long()
    kc = npy(inp["k_cache"][pages])
    vc = npy(inp["v_cache"][pages]) if inp.get("v_cache") is not None else None
    pt = np.arange(max(n, 1), dtype=np.int64)[None, :]
    return kc if n else np.zeros((1,) + tuple(inp["k_cache"].shape[1:]), np.float32), vc, pt, ctx


def oracle_attention_rows(inp, d_packed, cu, reqs):
    wl = inp["workload"]
    rows, o_all, l_all = [], [], []
    for r in reqs:
        c0, c1 = int(cu[r]), int(cu[r + 1])
        kc, vc, pt, ctx = sub_cache(inp, r)
        q = npy(d_packed["q"][c0:c1])
        kn = npy(d_packed["k_new"][c0:c1])
        sub_cu = np.array([0, c1 - c0])
        if wl.attn == "gqa":
            vn = npy(d_packed["v_new"][c0:c1])
            if vc is None:
                vc = np.zeros_like(kc)
            o, l = O.verify_attention_gqa(q, kn, vn, kc, vc, pt, np.array([ctx]), sub_cu, wl.Hq,
                                          wl.Hkv, 1.0 / math.sqrt(wl.d_qk))
        else:
            o, l = O.verify_attention_mla(q, kn, kc, pt, np.array([ctx]), sub_cu, wl.d_v,
                                          1.0 / math.sqrt(wl.d_qk))
        rows.extend(range(c0, c1))
        o_all.append(o)
        l_all.append(l)
    return rows, np.concatenate(o_all), np.concatenate(l_all)


def run_and_check(inp, mode, attention_requests=None):
    """Full step on the GPU, then every stage against the oracle."""
    wl = inp["workload"]
    snp = small_np(inp)
    d, step = harness.prepare(inp, mode)
    step.run(d, mode)
    err = harness.dspark.read_device_error()
    torch.cuda.synchronize()
    g = {
        "windows": step.windows.cpu(), "a_hat": step.a_hat.cpu(), "M": int(step.M.item()),
        "E": float(step.E.item()), "cu_seqlens": step.cu_seqlens.cpu(),
        "M_pack": int(step.M_pack.item()), "tier": int(step.tier.item()),
        "row_req": step.row_req.cpu(), "row_pos": step.row_pos.cpu(), "row_tok": step.row_tok.cpu(),
        "accept_len": step.accept_len.cpu(), "cap_len": step.cap_len.cpu(),
        "out_tok": step.out_tok.cpu(), "fallback": step.fallback.cpu(), "cstar": step.cstar.cpu(),
        "committed": step.committed.cpu(), "n_committed": step.n_committed.cpu(),
        "page_table": d["page_table"].cpu(), "ctx_len": d["ctx_len"].cpu(),
        "anchor": d["anchor"].cpu(), "free_top": int(d["free_top"].item()),
        "k_cache": d["k_cache"], "v_cache": d.get("v_cache"),
    }
    assert err == 0, f"device error word {err:#x}"
    sch = O.schedule(snp["conf"], inp["conf_is_logit"], snp["sts_temp"], snp["cost_table"],
                     wl.max_tokens, mode)
    windows = check_schedule(g, sch, wl.B)
    pk = O.pack(windows, snp["ctx_len"], snp["anchor"], snp["draft_tok"], snp["tiers"], mode,
                wl.gamma)
    check_pack(g, pk)
    M = pk.M
    reqs = range(wl.B) if attention_requests is None else attention_requests
    rows, o, l = oracle_attention_rows(inp, d, pk.cu_seqlens, reqs)
    check_attention(npy(step.out[rows]), npy(step.lse[rows]), o, l)
    p_t = npy(d["p_target"][:M])
    acc = O.accept(p_t, npy(inp["p_draft"]), snp["draft_tok"], snp["uniforms"],
                   npy(inp["exp_noise"]), windows, pk.cu_seqlens, mode, wl.gamma)
    check_accept(g, acc)
    cm = oracle_compact_state(snp, pk, acc, wl)
    check_compact(g, cm, inp, pk, acc, wl, d)
    return g, sch, pk, acc


# ------------------------------------------------------------------ tests

def test_smoke():
    import __graft_entry__ as g
    g.smoke()


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("mode", list(MODES))
def test_tiny_all_modes(seed, mode):
    inp = W.make_inputs(W.WORKLOADS["tiny"], seed)
    run_and_check(inp, MODES[mode])


def _edge_workload():
    return W.Workload(
        name="edges", B=8, gamma=5, attn="gqa", Hq=8, Hkv=2, d_qk=128, d_v=128, page_size=16,
        ctx=("const", 0), conf=("logit", 1.0, 1.0), vocab=1024, p_dtype="f32",
        target_logit_std=2.0, draft_noise_std=0.5, tiers=(8, 16, 32, 64), cost_theta_ms=0.05)


@pytest.mark.parametrize("mode", list(MODES))
def test_ragged_edges(mode):
    """ctx = 0, exactly one page, exactly one 64-key tile, several tiles with a ragged
    tail, a page boundary at the block; windows forced to 0 and to gamma."""
    wl = _edge_workload()
    inp = W.make_inputs(wl, seed=5, ctx_override=[0, 16, 64, 100, 257, 700, 1023, 47])
    conf = inp["conf"].clone()
    conf[0] = 20.0          # survives everything -> w = gamma
    conf[1] = -20.0         # survives nothing -> w = 0
    inp["conf"] = conf
    g, sch, pk, acc = run_and_check(inp, MODES[mode])
    if mode != "static":
        assert sch.windows[0] == wl.gamma and sch.windows[1] == 0


@pytest.mark.parametrize("mode", ["compact", "cap_accept"])
def test_all_zero_residual_falls_back_to_target(mode):
    """Draft = target everywhere except one inflated draft probability at request 0's
    first draft token, with u close to 1: that draft is rejected and the residual
    max(0, p_t - p_d) is zero on the whole row, so the correction is drawn from p_t
    (reading A12); every other request accepts its whole window."""
    wl = W.WORKLOADS["tiny"]
    inp = W.make_inputs(wl, 4)
    conf = inp["conf"].clone()
    conf[0] = 20.0                                   # request 0 verifies its whole block
    inp["conf"] = conf
    pd = inp["p_target_dense"][:, :wl.gamma].clone()
    x = int(inp["draft_tok"][0, 0])
    pd[0, 0, x] = pd[0, 0, x] * 1.5
    inp["p_draft"] = pd
    u = inp["uniforms"].clone()
    u[0, 0] = 0.99
    inp["uniforms"] = u
    g, sch, pk, acc = run_and_check(inp, MODES[mode])
    assert acc.residual_fallback[0] and int(acc.accept_len[0]) == 0


@pytest.mark.parametrize("B,G", [(3, 1), (5, 7), (2, 16)])
def test_group_sizes_and_row_tiles(B, G):
    """Query heads per KV head from 1 to 16 (16 x (gamma+1) > 128 rows: two row tiles)."""
    wl = W.Workload(
        name=f"g{G}", B=B, gamma=8, attn="gqa", Hq=2 * G, Hkv=2, d_qk=128, d_v=128, page_size=32,
        ctx=("uniform", 30, 300), conf=("logit", 3.0, 1.0), vocab=512, p_dtype="bf16",
        target_logit_std=2.0, draft_noise_std=0.5, tiers=(16, 32, 64), cost_theta_ms=0.01)
    inp = W.make_inputs(wl, seed=11)
    run_and_check(inp, O.STATIC)


@pytest.mark.parametrize("G,B", [(4, 6), (5, 5), (3, 7)])
def test_compact_windows_longer_than_the_query_tile(G, B):
    """Compact mode sizes the query tile for floor(32 / G) block rows; confident drafts
    make windows of up to gamma + 1 = 13 rows, so requests run as two or three row tiles
    of the 32-column tile, beside requests that fit one.  Every request's attention
    against fp64."""
    import speculative_decoding_verification_dspark_gb300 as dspark
    wl = W.Workload(
        name=f"rowtiles_g{G}", B=B, gamma=12, attn="gqa", Hq=2 * G, Hkv=2, d_qk=128, d_v=128,
        page_size=16, ctx=("uniform", 40, 700), conf=("logit", 3.0, 1.5), vocab=512,
        p_dtype="f32", target_logit_std=2.0, draft_noise_std=0.3, tiers=(32, 64, 128),
        cost_theta_ms=0.5)
    inp = W.make_inputs(wl, seed=5)
    hint = dspark.block_rows_hint_for(wl.gamma, wl.Hq, wl.Hkv, O.COMPACT)
    g, sch, pk, acc = run_and_check(inp, O.COMPACT)
    rows = np.diff(np.asarray(pk.cu_seqlens))
    assert hint == 32 // G
    assert int(rows.max()) > hint >= int(rows.min())  # split requests beside whole ones


def test_mla_small():
    wl = W.Workload(
        name="mla_small", B=3, gamma=4, attn="mla", Hq=128, Hkv=1, d_qk=576, d_v=512, page_size=64,
        ctx=("uniform", 40, 300), conf=("logit", 1.2, 1.0), vocab=1024, p_dtype="f32",
        target_logit_std=3.0, draft_noise_std=0.7, tiers=(8, 16))
    inp = W.make_inputs(wl, seed=3)
    run_and_check(inp, O.COMPACT)
    run_and_check(inp, O.STATIC)


def test_mla_page16_split():
    """Latent KV with 16-token pages (four TMA boxes per key tile) and contexts long
    enough that groups are cut into pieces across clusters."""
    wl = W.Workload(
        name="mla_p16", B=5, gamma=6, attn="mla", Hq=128, Hkv=1, d_qk=576, d_v=512, page_size=16,
        ctx=("uniform", 100, 2000), conf=("logit", 1.2, 1.0), vocab=1024, p_dtype="f32",
        target_logit_std=3.0, draft_noise_std=0.7, tiers=(8, 16, 32, 64))
    inp = W.make_inputs(wl, seed=5)
    run_and_check(inp, O.COMPACT)


@pytest.mark.parametrize("page_size,ctxs", [
    (32, [0, 32, 64, 100, 257, 700, 1023, 47]),
    (128, [0, 128, 64, 100, 257, 700, 1023, 47]),
    (64, [0, 64, 32, 33, 31, 97, 511, 1]),
])
def test_mla_ragged_edges(page_size, ctxs):
    """Latent KV: ctx = 0, exactly one page, one whole 64-key tile, a single key, keys
    just below, at and past half a tile, ragged tails and a page boundary at the block,
    with windows forced to gamma and to 0."""
    wl = W.Workload(
        name=f"mla_edges_p{page_size}", B=8, gamma=5, attn="mla", Hq=128, Hkv=1, d_qk=576,
        d_v=512, page_size=page_size, ctx=("const", 0), conf=("logit", 1.0, 1.0), vocab=1024,
        p_dtype="f32", target_logit_std=2.0, draft_noise_std=0.5, tiers=(8, 16, 32, 64),
        cost_theta_ms=0.05)
    inp = W.make_inputs(wl, seed=6, ctx_override=ctxs)
    conf = inp["conf"].clone()
    conf[0] = 20.0
    conf[1] = -20.0
    inp["conf"] = conf
    run_and_check(inp, O.COMPACT)


def _full(name, seed=0):
    wl = W.WORKLOADS[name]
    return W.make_inputs(wl, seed, device=W.gen_device(wl))


def test_full_qwen3_8b():
    """The timed shape, every request's attention against fp64 (all split groups and
    stream-K pieces of the timed launch configuration)."""
    inp = _full("qwen3_8b")
    run_and_check(inp, O.COMPACT)


@pytest.mark.parametrize("mode", list(MODES))
def test_full_mixed256(mode):
    """B=256, gamma=16: attention checked on 32 requests spread over the batch (all
    three confidence classes, short and long contexts)."""
    inp = _full("mixed256")
    run_and_check(inp, MODES[mode], attention_requests=list(range(0, 256, 8)))


def test_full_mla():
    """Latent-KV shape at full size: every request's attention against fp64."""
    inp = _full("mla")
    run_and_check(inp, O.COMPACT)


def _sweep_grid():
    """Points of the budget/tier sweep: every (confidence mean, cost slope) pair once,
    the batch sizes taken in turn, plus the largest batch at every confidence mean."""
    pts = []
    i = 0
    for c in W.SWEEP_CONF_MEANS:
        for theta in W.SWEEP_THETA:
            pts.append((W.SWEEP_B[i % len(W.SWEEP_B)], c, theta))
            i += 1
    for c in W.SWEEP_CONF_MEANS:
        pts.append((256, c, 0.19))
    return pts


@pytest.mark.parametrize("B,c,theta", _sweep_grid())
def test_sweep_points(B, c, theta):
    wl = W.sweep_point(B, c, theta)
    inp = W.make_inputs(wl, 0, device=W.gen_device(wl))
    for mode in (O.COMPACT, O.STATIC, O.CAP_ACCEPT):
        run_and_check(inp, mode, attention_requests=sorted({0, B // 2, B - 1}))


# ------------------------------------------------------------------ peaked softmax

def _peaked(inp, factor):
    """Queries scaled by a power of two (exact in bf16): logits of standard deviation
    `factor`, so a few keys carry most of the softmax mass.  This is where the bf16
    rounding of P, the deferred rescale of the output accumulator and (latent KV) the
    exchange of partial scores between the two CTAs of a cluster matter."""
    inp = dict(inp)
    inp["q_dense"] = (inp["q_dense"].float() * factor).to(torch.bfloat16)
    return inp


@pytest.mark.parametrize("factor,gamma,mode", [(8, 8, "compact"), (16, 8, "compact"),
                                               (8, 16, "static"), (16, 16, "cap_accept")])
def test_peaked_softmax_gqa(factor, gamma, mode):
    """GQA with peaked scores; gamma = 16 in static/cap-accept mode puts 17 rows x 4
    heads on the 128-column query tile."""
    wl = W.Workload(
        name=f"peaked_gqa_g{gamma}", B=6, gamma=gamma, attn="gqa", Hq=32, Hkv=8, d_qk=128,
        d_v=128, page_size=16, ctx=("uniform", 700, 3000), conf=("logit", 1.5, 1.0), vocab=1024,
        p_dtype="f32", target_logit_std=3.0, draft_noise_std=0.7,
        tiers=W.pow2_tiers(8, 6 * (gamma + 1)))
    inp = _peaked(W.make_inputs(wl, 21), factor)
    run_and_check(inp, MODES[mode])


@pytest.mark.parametrize("factor,page_size", [(4, 64), (8, 64), (8, 16)])
def test_peaked_softmax_mla(factor, page_size):
    """Latent KV with peaked scores (standard deviation 4 or 8 instead of 1)."""
    wl = W.Workload(
        name=f"peaked_mla_p{page_size}", B=4, gamma=6, attn="mla", Hq=128, Hkv=1, d_qk=576,
        d_v=512, page_size=page_size, ctx=("uniform", 1000, 6000), conf=("logit", 1.2, 1.0),
        vocab=1024, p_dtype="f32", target_logit_std=3.0, draft_noise_std=0.7,
        tiers=(8, 16, 32))
    inp = _peaked(W.make_inputs(wl, 22), factor)
    run_and_check(inp, O.COMPACT)


# ------------------------------------------------------------------ crafted acceptance

def _accept_direct(p_t, p_d, draft, u, e, windows, cu, mode):
    """dspark_accept on crafted host tensors; returns the GPU outputs (host)."""
    import speculative_decoding_verification_dspark_gb300 as dspark
    dev = torch.device("cuda")
    B, gamma, V = p_d.shape
    i32 = dict(dtype=torch.int32, device=dev)
    t = {k: torch.as_tensor(v).to(dev) for k, v in dict(p_t=p_t, p_d=p_d, e=e, u=u).items()}
    draft_d = torch.as_tensor(draft, dtype=torch.int32).to(dev)
    win_d = torch.as_tensor(windows, dtype=torch.int32).to(dev)
    cu_d = torch.as_tensor(cu, dtype=torch.int32).to(dev)
    out = {"accept_len": torch.full((B,), -7, **i32), "cap_len": torch.full((B,), -7, **i32),
           "out_tok": torch.full((B,), -7, **i32), "fallback": torch.full((B,), -7, **i32),
           "cstar": torch.full((B, gamma), 3.0, dtype=torch.float32, device=dev)}
    ws = torch.empty(dspark.accept_workspace_size(B, gamma, p_t.shape[0], V), dtype=torch.uint8,
                     device=dev)
    dspark.read_device_error()
    dspark.accept(t["p_t"], t["p_d"], draft_d, t["u"], t["e"], win_d, cu_d, mode,
                  out["accept_len"], out["cap_len"], out["out_tok"], out["cstar"],
                  out["fallback"], ws)
    torch.cuda.synchronize()
    assert dspark.read_device_error() == 0
    return {k: v.cpu() for k, v in out.items()}


@pytest.mark.parametrize("maxima", [
    [36, 37, 300, 8193, 8200, 20000],      # same lane, other warps, later chunks
    [20000, 8200, 4100, 4099],              # lowest in the first chunk, last warps
    [24000, 16384, 8192],                   # chunk boundaries only
    [25575, 12345],                          # last entry of the vocabulary
])
@pytest.mark.parametrize("dtype", [np.float32, "bf16"])
def test_race_ties_lowest_index_on_gpu(maxima, dtype):
    """The largest race key duplicated across lanes, warps and 8192-entry chunks: the
    lowest index wins, on a bonus row (request 0) and on a correction row (request 1);
    request 2 tests u * p_d = p_t exactly (accepted: the test is inclusive) followed by
    p_t one ulp below u * p_d (rejected)."""
    V, gamma, B = 3 * 8192 + 1000, 4, 3
    rng = np.random.default_rng(sum(maxima))
    n = gamma + 1
    cu = np.arange(B + 1, dtype=np.int32) * n
    p_t = rng.uniform(1e-6, 1e-4, size=(B * n, V)).astype(np.float32)
    p_d = rng.uniform(1e-6, 1e-4, size=(B, gamma, V)).astype(np.float32)
    e = rng.uniform(1.0, 2.0, size=(B, V)).astype(np.float32)
    draft = np.zeros((B, gamma), np.int32)
    u = np.full((B, gamma), 2.0 ** -20, np.float32)
    # request 0: every draft accepted (u tiny), bonus drawn on row 4 from p_t
    for j in range(gamma):
        draft[0, j] = 11 + j
    for m in maxima:
        p_t[cu[0] + gamma, m] = 0.5
        e[0, m] = 1.0
    # request 1: draft 1 rejected (p_t = 0 there), correction from max(0, p_t - p_d) on
    # row 0 with the maximal residual 0.25 at the duplicated indices
    draft[1, 0] = 77
    p_t[cu[1], 77] = 0.0
    for m in maxima:
        p_t[cu[1], m] = 0.375
        p_d[1, 0, m] = 0.125
        e[1, m] = 1.0
    # request 2: u * p_d == p_t exactly at positions 1, 2; one ulp below at 3
    u[2] = 0.75
    for j, x in enumerate((5, 6, 7)):
        draft[2, j] = x
        p_d[2, j, x] = 0.5
        p_t[cu[2] + j, x] = 0.375 if j < 2 else np.nextafter(np.float32(0.375), np.float32(0))
    windows = np.full(B, gamma, np.int32)
    if dtype == "bf16":
        # (bf16 cannot hold 0.375 minus one fp32 ulp: there request 2 accepts on)
        pt_d = torch.from_numpy(p_t).to(torch.bfloat16)
        pd_d = torch.from_numpy(p_d).to(torch.bfloat16)
        pt_o, pd_o = pt_d.float().numpy(), pd_d.float().numpy()
    else:
        pt_d, pd_d = p_t, p_d
        pt_o, pd_o = p_t, p_d
    g = _accept_direct(pt_d, pd_d, draft, u, e, windows, cu, O.COMPACT)
    acc = O.accept(pt_o, pd_o, draft, u, e, windows, cu, O.COMPACT, gamma)
    assert acc.accept_len.tolist()[:2] == [gamma, 0]
    assert acc.accept_len[2] >= 2 and (dtype == "bf16" or acc.accept_len[2] == 2)
    assert acc.out_tok[0] == min(maxima) and acc.out_tok[1] == min(maxima)
    assert np.array_equal(g["accept_len"].numpy(), acc.accept_len)
    assert np.array_equal(g["cap_len"].numpy(), acc.cap_len)
    assert np.array_equal(g["out_tok"].numpy(), acc.out_tok)
    assert np.array_equal(g["fallback"].numpy().astype(bool), acc.residual_fallback)
    cs = g["cstar"].numpy()
    assert np.nanmax(np.abs(cs - acc.cstar)) <= CSTAR_TOL


def test_race_zero_weights_with_zero_noise_on_gpu():
    """Zero noise entries placed on zero weights (their w / e is NaN), and a row whose
    only positive residual entries carry large noise: the zero-weight entries never
    win, on the GPU as in the oracle (reading A11)."""
    V, gamma, B = 2 * 8192 + 64, 2, 2
    rng = np.random.default_rng(5)
    n = gamma + 1
    cu = np.arange(B + 1, dtype=np.int32) * n
    p_t = rng.uniform(0.0, 1e-4, size=(B * n, V)).astype(np.float32)
    p_d = rng.uniform(0.0, 1e-4, size=(B, gamma, V)).astype(np.float32)
    e = rng.uniform(0.5, 2.0, size=(B, V)).astype(np.float32)
    draft = np.array([[3, 4], [9, 10]], np.int32)
    u = np.full((B, gamma), 2.0 ** -20, np.float32)
    # request 0: bonus row with zero weights and zero noise on every 7th entry
    zero = np.arange(0, V, 7)
    p_t[cu[0] + gamma, zero] = 0.0
    e[0, zero] = 0.0
    # request 1: rejected at position 1; residual positive only at 3 entries, the rest
    # zero, and zero noise on many zero-residual entries
    p_t[cu[1], 9] = 0.0
    p_d[1, 0] = p_t[cu[1]] + np.float32(1e-3)
    for m, ev in ((100, 1e6), (9000, 3e6), (16000, 2e6)):
        p_t[cu[1], m] = 0.01
        p_d[1, 0, m] = 0.005
        e[1, m] = ev
    e[1, np.arange(1, V, 5)] = 0.0
    e[1, [100, 9000, 16000]] = [1e6, 3e6, 2e6]
    windows = np.full(B, gamma, np.int32)
    g = _accept_direct(p_t, p_d, draft, u, e, windows, cu, O.COMPACT)
    acc = O.accept(p_t, p_d, draft, u, e, windows, cu, O.COMPACT, gamma)
    assert acc.out_tok[1] == 100 and not acc.residual_fallback[1]
    assert acc.out_tok[0] % 7 != 0
    assert np.array_equal(g["out_tok"].numpy(), acc.out_tok)
    assert np.array_equal(g["accept_len"].numpy(), acc.accept_len)
    assert np.array_equal(g["fallback"].numpy().astype(bool), acc.residual_fallback)


def test_cap_accept_commits_match_compact_on_gpu():
    inp = _full("mixed256", seed=1)
    outs = {}
    for mode in (O.COMPACT, O.CAP_ACCEPT):
        d, step = harness.prepare(inp, mode)
        step.run(d, mode)
        torch.cuda.synchronize()
        outs[mode] = (step.accept_len.cpu(), step.out_tok.cpu(), step.committed.cpu(),
                      d["page_table"].cpu())
    for a, b in zip(outs[O.COMPACT], outs[O.CAP_ACCEPT]):
        assert torch.equal(a, b)


def test_deterministic_bytes():
    inp = _full("qwen3_8b", seed=2)
    res = []
    for _ in range(2):
        d, step = harness.prepare(inp, O.COMPACT)
        step.run(d, O.COMPACT)
        torch.cuda.synchronize()
        res.append([step.out.clone(), step.lse.clone(), step.cstar.clone(), step.out_tok.clone(),
                    d["k_cache"].clone()])
    for a, b in zip(*res):
        assert torch.equal(a.view(torch.uint8) if a.dtype != torch.int32 else a,
                           b.view(torch.uint8) if b.dtype != torch.int32 else b)


def test_free_stack_exhausted_sets_error_and_changes_nothing():
    import speculative_decoding_verification_dspark_gb300 as dspark
    wl = W.WORKLOADS["tiny"]
    inp = W.make_inputs(wl, 0, extra_free_pages=0, ctx_override=[64, 80, 96, 128])
    d, step = harness.prepare(inp, O.COMPACT)
    before = harness.snapshot_state(d)
    dspark.read_device_error()
    step.run(d, O.COMPACT)
    err = dspark.read_device_error()
    assert err & 0x2
    for k, v in before.items():
        if isinstance(v, torch.Tensor):
            assert torch.equal(d[k], v), k


def test_rows_overflow_is_reported():
    import speculative_decoding_verification_dspark_gb300 as dspark
    wl = W.WORKLOADS["tiny"]
    inp = W.make_inputs(wl, 0)
    d = harness.device_inputs(inp)
    step = dspark.VerifyStep(wl.B, wl.gamma, wl.Hq, wl.Hkv, wl.d_qk, wl.d_v, wl.vocab, max_rows=4)
    dspark.read_device_error()
    step.schedule(d, O.STATIC)
    step.pack(d, O.STATIC)
    assert dspark.read_device_error() & 0x1
    # the later stages see packed rows beyond their 4-row buffers: each one reports
    # the overflow and reads or writes no row (the state is left as it was)
    assert int(step.cu_seqlens[-1]) > 4
    dev = torch.device("cuda")
    d["q"] = torch.zeros(4, wl.Hq, wl.d_qk, dtype=torch.bfloat16, device=dev)
    d["k_new"] = torch.zeros(4, wl.Hkv, wl.d_qk, dtype=torch.bfloat16, device=dev)
    d["v_new"] = torch.zeros(4, wl.Hkv, wl.d_v, dtype=torch.bfloat16, device=dev)
    d["p_target"] = torch.zeros(4, wl.vocab, dtype=torch.float32, device=dev)
    before = harness.snapshot_state(d)
    for run in (lambda: step.attention(d), lambda: step.accept(d, O.STATIC),
                lambda: step.compact(d)):
        run()
        assert dspark.read_device_error() & 0x1
    for k, v in before.items():
        if isinstance(v, torch.Tensor):
            assert torch.equal(d[k], v), k
    # the same through the fused pack + work list and the planned attention
    step.pack_plan(d, O.STATIC)
    assert dspark.read_device_error() & 0x1
    step.attention_planned(d)
    assert dspark.read_device_error() & 0x1
    for k, v in before.items():
        if isinstance(v, torch.Tensor):
            assert torch.equal(d[k], v), k


@pytest.mark.parametrize("shape", ["gqa", "mla"])
def test_planned_attention_equals_standalone(shape):
    """The work list built inside the pack kernel is the attention call's own: the planned
    attention gives the standalone call's outputs bit for bit."""
    if shape == "gqa":
        wl = W.WORKLOADS["tiny"]
        inp = W.make_inputs(wl, 4)
    else:
        wl = W.Workload(
            name="mla_plan", B=5, gamma=6, attn="mla", Hq=128, Hkv=1, d_qk=576, d_v=512,
            page_size=16, ctx=("uniform", 100, 2000), conf=("logit", 1.2, 1.0), vocab=1024,
            p_dtype="f32", target_logit_std=3.0, draft_noise_std=0.7, tiers=(8, 16, 32, 64))
        inp = W.make_inputs(wl, 7)
    d, step = harness.prepare(inp, O.COMPACT)
    M = int(step.cu_seqlens[-1])
    step.attention(d)
    torch.cuda.synchronize()
    out0, lse0 = step.out[:M].clone(), step.lse[:M].clone()
    step.out.zero_()
    step.lse.zero_()
    step.pack_plan(d, O.COMPACT)
    step.attention_planned(d)
    torch.cuda.synchronize()
    assert torch.equal(step.out[:M], out0)
    assert torch.equal(step.lse[:M], lse0)


@pytest.mark.parametrize("windows", [[3, 2, 1], [3, 2, 2], [6, 6, 6], [0]])
def test_pack_tier_edges_on_gpu(windows):
    """M equal to a tier, one row past it, above every tier, and a single anchor-only
    request: the pack call and the pack + work list call both give the oracle's rows."""
    import speculative_decoding_verification_dspark_gb300 as dspark
    gamma, B, max_rows = 6, len(windows), 32
    tiers = [4, 9, 16]
    dev = torch.device("cuda")
    i32 = dict(dtype=torch.int32, device=dev)
    w = torch.tensor(windows, **i32)
    ctx = torch.tensor([0, 16, 100][:B], **i32)
    anchor = torch.tensor([5, 6, 7][:B], **i32)
    drafts = torch.arange(B * gamma, **i32).reshape(B, gamma)
    tiers_d = torch.tensor(tiers, **i32)
    pk = O.pack(np.array(windows, np.int32), ctx.cpu().numpy(), anchor.cpu().numpy(),
                drafts.cpu().numpy(), tiers, O.COMPACT, gamma)
    ws = torch.empty(dspark.verify_attn_workspace_size(B, max_rows, 8, 2, 128, 128, 8, gamma + 1),
                     dtype=torch.uint8, device=dev)
    dspark.read_device_error()
    for fused in (False, True):
        cu, M, tier = torch.zeros(B + 1, **i32), torch.zeros(1, **i32), torch.zeros(1, **i32)
        rr, rp, rt = (torch.full((max_rows,), 99, **i32) for _ in range(3))
        if fused:
            dspark.pack_plan(w, ctx, anchor, drafts, tiers_d, O.COMPACT, cu, M, tier, rr, rp, rt,
                             8, 2, 128, 128, max_rows, 8, ws, max_block_rows=gamma + 1)
        else:
            dspark.pack(w, ctx, anchor, drafts, tiers_d, O.COMPACT, cu, M, tier, rr, rp, rt)
        torch.cuda.synchronize()
        assert cu.cpu().numpy().tolist() == pk.cu_seqlens.tolist()
        assert int(M) == pk.M and int(tier) == pk.tier
        T = pk.tier
        assert rr.cpu().numpy()[:T].tolist() == pk.row_req.tolist()
        assert rp.cpu().numpy()[:T].tolist() == pk.row_pos.tolist()
        assert rt.cpu().numpy()[:T].tolist() == pk.row_tok.tolist()
        assert rr.cpu().numpy()[T:].tolist() == [99] * (max_rows - T)  # rows past the tier untouched
        assert dspark.read_device_error() == 0

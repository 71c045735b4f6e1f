"""The device-resident step: the pinned tier word of the pack call, and the step
graph (tier chosen on the device by a switch node) replayed over a chain of steps
whose tiers change, with no host synchronisation between the steps.  Every step
of the chain is compared with the oracle's chain (state carried over by its own
compaction), and with the same chain run through the five calls one by one."""
import math

import numpy as np
import pytest
import torch

import harness
import workloads as W
from oracle import dspark_oracle as O

pytestmark = pytest.mark.gpu

ATT_MAX, ATT_MEAN, LSE_MAX, CSTAR_TOL = 1e-2, 1e-3, 4e-3, 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _npy(t):
    t = t.detach().cpu()
    return (t.float() if t.dtype == torch.bfloat16 else t).numpy()


def test_pinned_tier_word_without_stream_sync():
    """The pack kernel stores the tier into a pinned, mapped host word; after an event
    recorded behind the pack call has completed, the host reads it there."""
    import speculative_decoding_verification_dspark_gb300 as dspark
    wl = W.WORKLOADS["tiny"]
    inp = W.make_inputs(wl, 2)
    d = harness.device_inputs(inp)
    step = harness.make_step(wl)
    tier_host = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        step.schedule(d, O.COMPACT)
        for fused in (False, True):
            tier_host.fill_(-1)
            if fused:
                dspark.pack_plan(step.windows, d["ctx_len"], d["anchor"], d["draft_tok"],
                                 d["tiers"], O.COMPACT, step.cu_seqlens, step.M_pack, step.tier,
                                 step.row_req, step.row_pos, step.row_tok, wl.Hq, wl.Hkv, wl.d_qk,
                                 wl.d_v, step.max_rows, step.max_splits, step.ws_attn,
                                 max_block_rows=wl.gamma + 1, tier_host=tier_host)
            else:
                dspark.pack(step.windows, d["ctx_len"], d["anchor"], d["draft_tok"], d["tiers"],
                            O.COMPACT, step.cu_seqlens, step.M_pack, step.tier, step.row_req,
                            step.row_pos, step.row_tok, tier_host=tier_host)
            ev = torch.cuda.Event()
            ev.record(stream)
            ev.synchronize()
            sch = O.schedule(_npy(inp["conf"]), inp["conf_is_logit"], _npy(inp["sts_temp"]),
                             _npy(inp["cost_table"]), wl.max_tokens, O.COMPACT)
            pk = O.pack(sch.windows, _npy(inp["ctx_len"]), _npy(inp["anchor"]),
                        _npy(inp["draft_tok"]), list(wl.tiers), O.COMPACT, wl.gamma)
            assert int(tier_host[0]) == pk.tier
    torch.cuda.synchronize()
    assert int(step.tier[0]) == pk.tier
    assert dspark.read_device_error() == 0


def _chain(wl, n_steps, seed, shifts):
    """Inputs of a chain of steps: the cache, page table and free stack of one draw
    (with room for the chain's growth), and per step fresh drafter/target tensors
    whose confidence logits are shifted by shifts[k] (so the windows, M and the tier
    change from step to step)."""
    base = W.make_inputs(wl, seed, extra_free_pages=wl.B * n_steps * 2)
    grow = (n_steps * (wl.gamma + 1) + wl.page_size - 1) // wl.page_size + 1
    pt = base["page_table"]
    base["page_table"] = torch.cat(
        [pt, torch.full((wl.B, grow), -1, dtype=torch.int32)], dim=1).contiguous()
    steps = []
    for k in range(n_steps):
        s = W.make_inputs(wl, seed * 100 + k + 1)
        s["conf"] = (s["conf"].double() + shifts[k % len(shifts)]).float()
        steps.append(s)
    return base, steps


STEP_KEYS = ("conf", "draft_tok", "p_draft", "uniforms", "exp_noise")
ROW_KEYS = ("q", "k_new", "v_new", "p_target")
DENSE = {"q": "q_dense", "k_new": "k_new_dense", "v_new": "v_new_dense",
         "p_target": "p_target_dense"}


def _oracle_chain(wl, base, steps, mode):
    """The oracle over the chain; the state after each step feeds the next."""
    st = {k: _npy(base[k]) for k in ("page_table", "ctx_len", "anchor", "k_cache", "v_cache",
                                      "free_pages")}
    st["free_top"] = int(base["free_top"][0])
    res = []
    for s in steps:
        sch = O.schedule(_npy(s["conf"]), s["conf_is_logit"], _npy(s["sts_temp"]),
                         _npy(s["cost_table"]), wl.max_tokens, mode)
        assert not sch.listed, "chain inputs with a near-margin window decision"
        pk = O.pack(sch.windows, st["ctx_len"], st["anchor"], _npy(s["draft_tok"]),
                    list(wl.tiers), mode, wl.gamma)
        cu = torch.as_tensor(pk.cu_seqlens)
        packed = {k: W.to_packed(s[DENSE[k]], cu, W.cap_rows(wl)) for k in ROW_KEYS}
        pn = {k: _npy(v) for k, v in packed.items()}
        o, lse = O.verify_attention_gqa(pn["q"], pn["k_new"], pn["v_new"], st["k_cache"],
                                        st["v_cache"], st["page_table"], st["ctx_len"],
                                        pk.cu_seqlens, wl.Hq, wl.Hkv, 1.0 / math.sqrt(wl.d_qk))
        acc = O.accept(pn["p_target"][:pk.M], _npy(s["p_draft"]), _npy(s["draft_tok"]),
                       _npy(s["uniforms"]), _npy(s["exp_noise"]), sch.windows, pk.cu_seqlens,
                       mode, wl.gamma)
        cm = O.compact(pn["k_new"], pn["v_new"], pk.cu_seqlens, acc.accept_len, acc.out_tok,
                       _npy(s["draft_tok"]), wl.page_size, st["page_table"], st["ctx_len"],
                       st["anchor"], st["free_pages"], st["free_top"], st["k_cache"],
                       st["v_cache"])
        res.append({"sch": sch, "pk": pk, "o": o, "lse": lse, "acc": acc, "cm": cm,
                    "packed": packed})
        st.update(page_table=cm.page_table, ctx_len=cm.ctx_len, anchor=cm.anchor,
                  k_cache=cm.k_cache, v_cache=cm.v_cache, free_top=cm.free_top)
    return res


OUT_KEYS = ("windows", "cu_seqlens", "tier", "out", "lse", "accept_len", "cap_len", "out_tok",
            "cstar", "committed", "n_committed")
STATE_KEYS = ("page_table", "ctx_len", "anchor", "free_top")


def _run_chain(wl, base, steps, ora, mode, use_graph):
    """The chain on the GPU: per step, the step's inputs are copied into the fixed
    buffers (device to device, on the stream), one step runs (the step graph, or
    the five calls), and its outputs are copied aside; the host reads nothing until
    the end."""
    import speculative_decoding_verification_dspark_gb300 as dspark
    d = harness.device_inputs(base)
    step = harness.make_step(wl)
    dev = step.windows.device
    # the fixed input buffers the graph is built on
    for k in STEP_KEYS:
        d[k] = steps[0][k].to(dev).contiguous()
    for k in ROW_KEYS:
        d[k] = ora[0]["packed"][k].to(dev).contiguous()
    stash = [{**{k: s[k].to(dev) for k in STEP_KEYS},
              **{k: r["packed"][k].to(dev) for k in ROW_KEYS}} for s, r in zip(steps, ora)]
    n = len(steps)
    log = torch.zeros(1 + n, dtype=torch.int32, device=dev)
    tier_host = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    g = step.graph(d, mode, tier_host=tier_host, body_log=log) if use_graph else None
    dspark.read_device_error()
    outs = []
    stream = torch.cuda.current_stream()
    for k in range(n):
        for key, v in stash[k].items():
            d[key].copy_(v, non_blocking=True)
        if use_graph:
            g.launch(stream)
        else:
            step.run(d, mode)
        outs.append({**{key: getattr(step, key).clone() for key in OUT_KEYS},
                     **{key: d[key].clone() for key in STATE_KEYS}})
    torch.cuda.synchronize()
    err = dspark.read_device_error()
    final = {"k_cache": d["k_cache"].clone(), "v_cache": d["v_cache"].clone()}
    body = log.cpu().numpy()
    if g is not None:
        g.close()
    return outs, final, body, err, int(tier_host[0])


@pytest.mark.parametrize("mode", ["compact", "cap_accept"])
def test_step_graph_chain_with_changing_tiers(mode):
    mode = W.MODE_NAMES[mode]
    wl = W.WORKLOADS["tiny"]
    n = 6
    base, steps = _chain(wl, n, 3, shifts=[4.0, -3.0, 0.5, -6.0, 6.0, 1.0])
    ora = _oracle_chain(wl, base, steps, mode)
    tiers_seen = [r["pk"].tier for r in ora]
    if mode == O.COMPACT:
        assert len(set(tiers_seen)) >= 2, tiers_seen   # the chain really changes tier
    outs, final, body, err, tier_last = _run_chain(wl, base, steps, ora, mode, use_graph=True)
    assert err == 0, f"device error word {err:#x}"
    # the switch ran the body of each step's tier (device-side choice), one per launch
    tiers = list(wl.tiers)
    assert body[0] == n
    assert body[1:].tolist() == [tiers.index(t) if t in tiers else len(tiers) for t in tiers_seen]
    assert tier_last == tiers_seen[-1]
    for k, (g, r) in enumerate(zip(outs, ora)):
        pk, acc, cm = r["pk"], r["acc"], r["cm"]
        assert np.array_equal(g["windows"].cpu().numpy(), r["sch"].windows), k
        assert np.array_equal(g["cu_seqlens"].cpu().numpy(), pk.cu_seqlens), k
        assert int(g["tier"][0]) == pk.tier, k
        M = pk.M
        err_o = np.abs(_npy(g["out"][:M]) - r["o"])
        assert err_o.max() <= ATT_MAX and err_o.mean() <= ATT_MEAN, (k, err_o.max())
        assert np.abs(_npy(g["lse"][:M]) - r["lse"]).max() <= LSE_MAX, k
        assert np.array_equal(g["accept_len"].cpu().numpy(), acc.accept_len), k
        assert np.array_equal(g["cap_len"].cpu().numpy(), acc.cap_len), k
        assert np.array_equal(g["out_tok"].cpu().numpy(), acc.out_tok), k
        cs = _npy(g["cstar"])
        assert np.array_equal(np.isnan(cs), np.isnan(acc.cstar)), k
        assert np.nanmax(np.abs(cs - acc.cstar)) <= CSTAR_TOL, k
        assert np.array_equal(g["committed"].cpu().numpy(), cm.committed), k
        assert np.array_equal(g["page_table"].cpu().numpy(), cm.page_table), k
        assert np.array_equal(g["ctx_len"].cpu().numpy(), cm.ctx_len), k
        assert np.array_equal(g["anchor"].cpu().numpy(), cm.anchor), k
        assert int(g["free_top"][0]) == cm.free_top, k
    assert np.array_equal(_npy(final["k_cache"]), ora[-1]["cm"].k_cache)
    assert np.array_equal(_npy(final["v_cache"]), ora[-1]["cm"].v_cache)
    # the same chain through the five calls: bit-identical
    outs2, final2, _, err2, _ = _run_chain(wl, base, steps, ora, mode, use_graph=False)
    assert err2 == 0
    def same_bits(x, y):  # NaN-aware: compares the bytes
        return torch.equal(x.contiguous().view(torch.uint8), y.contiguous().view(torch.uint8))

    for a, b in zip(outs, outs2):
        for key in a:
            assert same_bits(a[key], b[key]), key
    assert same_bits(final["k_cache"], final2["k_cache"])

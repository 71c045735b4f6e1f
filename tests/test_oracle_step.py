"""Whole-step invariants of the oracle on the tiny workload (CPU)."""
import numpy as np
import pytest

import workloads as W
from oracle import dspark_oracle as O
from helpers import oracle_step


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_cap_accept_commits_what_compact_commits(seed):
    inp = W.make_inputs(W.WORKLOADS["tiny"], seed)
    c, _ = oracle_step(inp, O.COMPACT, with_attention=False)
    k, _ = oracle_step(inp, O.CAP_ACCEPT, with_attention=False)
    assert np.array_equal(c["accept"].accept_len, k["accept"].accept_len)
    assert np.array_equal(c["accept"].out_tok, k["accept"].out_tok)
    assert np.all(k["accept"].cap_len >= k["accept"].accept_len)
    assert np.array_equal(c["compact"].page_table, k["compact"].page_table)
    assert np.array_equal(c["compact"].committed, k["compact"].committed)
    # the compacted cache holds the same rows: the segments differ only in length
    assert np.array_equal(c["compact"].k_cache, k["compact"].k_cache)


@pytest.mark.parametrize("seed", [0, 1])
def test_static_equals_full_window_compact(seed):
    wl = W.WORKLOADS["tiny"]
    inp = W.make_inputs(wl, seed)
    s, _ = oracle_step(inp, O.STATIC, with_attention=False)
    assert np.all(s["schedule"].windows == wl.gamma)
    # compact mode with a zero-slope cost table and room for everything verifies the whole block
    inp2 = dict(inp)
    inp2["cost_table"] = inp["cost_table"] * 0 + 20.0
    inp2["workload"] = wl.replace(tiers=(64,))
    c, _ = oracle_step(inp2, O.COMPACT, with_attention=False)
    assert np.all(c["schedule"].windows == wl.gamma)
    for f in ("accept_len", "cap_len", "out_tok"):
        assert np.array_equal(getattr(s["accept"], f), getattr(c["accept"], f))
    assert np.allclose(s["accept"].cstar, c["accept"].cstar, equal_nan=True)


def test_tiny_step_runs_with_attention():
    inp = W.make_inputs(W.WORKLOADS["tiny"], 0)
    out, packed = oracle_step(inp, O.COMPACT)
    o, lse = out["attn"]
    M = out["pack"].M
    assert o.shape[0] == M and np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    assert out["compact"].free_top <= int(inp["free_top"][0])

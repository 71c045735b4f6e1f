"""Host-side helpers of bench.py on CPU: the one-copy restore of the step's small
mutable state, and which sources a committed DRAM-traffic figure is keyed to."""
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402

KEYS = ("page_table", "ctx_len", "anchor", "free_top")


def _state():
    g = torch.Generator().manual_seed(3)
    return {
        "page_table": torch.randint(-1, 500, (5, 7), generator=g, dtype=torch.int32),
        "ctx_len": torch.randint(0, 900, (5,), generator=g, dtype=torch.int32),
        "anchor": torch.randint(0, 1000, (5,), generator=g, dtype=torch.int32),
        "free_top": torch.tensor([123], dtype=torch.int32),
    }


def test_restore_pairs_is_one_copy_of_views():
    d = _state()
    before = {k: v.clone() for k, v in d.items()}
    pairs = bench.restore_pairs(d, KEYS)
    assert len(pairs) == 1
    flat, saved = pairs[0]
    for k in KEYS:
        assert torch.equal(d[k], before[k]) and d[k].shape == before[k].shape
        assert d[k].is_contiguous()
        assert d[k].untyped_storage().data_ptr() == flat.untyped_storage().data_ptr()
        assert (d[k].data_ptr() - flat.data_ptr()) % 256 == 0  # each view on a 256-byte boundary
    # the step mutates the state in place; one copy puts all of it back
    d["page_table"].fill_(-7)
    d["ctx_len"] += 5
    d["anchor"].zero_()
    d["free_top"][0] = 0
    for dst, src in pairs:
        dst.copy_(src)
    for k in KEYS:
        assert torch.equal(d[k], before[k])
    assert not torch.equal(saved, torch.zeros_like(saved))


def test_restore_pairs_falls_back_on_mixed_dtypes():
    d = _state()
    d["anchor"] = d["anchor"].to(torch.int64)
    before = {k: v.clone() for k, v in d.items()}
    pairs = bench.restore_pairs(d, KEYS)
    assert len(pairs) == len(KEYS)
    for k in KEYS:
        d[k].zero_()
    for dst, src in pairs:
        dst.copy_(src)
    for k in KEYS:
        assert torch.equal(d[k], before[k])


def test_traffic_sources_follow_the_head_shape():
    gqa = {os.path.basename(p) for p in bench.attn_src(W.WORKLOADS["qwen3_8b"])}
    mla = {os.path.basename(p) for p in bench.attn_src(W.WORKLOADS["mla"])}
    assert "verify_attn_gqa.cu" in gqa and "verify_attn_mla.cu" not in gqa
    assert "verify_attn_mla.cu" in mla and "verify_attn_gqa.cu" not in mla
    assert {"verify_attn.cu", "worklist.cuh", "attn.h", "ptx.cuh", "common.cuh"} <= gqa & mla
    for p in bench.attn_src(W.WORKLOADS["mla"]) + bench.ACCEPT_SRC:
        assert os.path.isfile(p), p


def test_query_tile_policy():
    """Compact mode sizes the attention's query tile for floor(32 / G) block rows (the
    32-column tile), static and cap-accept for the whole block; the traffic key names
    the tile each selects."""
    import speculative_decoding_verification_dspark_gb300 as dspark
    q = W.WORKLOADS["qwen3_8b"]                     # G = 4, gamma = 8
    assert dspark.block_rows_hint_for(q.gamma, q.Hq, q.Hkv, dspark.COMPACT) == 8
    assert dspark.block_rows_hint_for(q.gamma, q.Hq, q.Hkv, dspark.STATIC) == 9
    assert dspark.block_rows_hint_for(q.gamma, q.Hq, q.Hkv, dspark.CAP_ACCEPT) == 9
    assert bench.query_tile(q, 8) == "nt32" and bench.query_tile(q, 9) == "nt64"
    m = W.WORKLOADS["mixed256"]                     # G = 5, gamma = 16
    assert dspark.block_rows_hint_for(m.gamma, m.Hq, m.Hkv, dspark.COMPACT) == 6
    assert bench.query_tile(m, 6) == "nt32" and bench.query_tile(m, 17) == "nt128"
    t = W.WORKLOADS["tiny"]                         # the whole block already fits 32 columns
    assert dspark.block_rows_hint_for(t.gamma, t.Hq, t.Hkv, dspark.COMPACT) == t.gamma + 1
    assert dspark.block_rows_hint_for(8, 64, 8, dspark.COMPACT) == 4    # G = 8: 32 columns
    assert dspark.block_rows_hint_for(8, 32, 2, dspark.COMPACT) == 4    # G = 16: 64 columns
    assert dspark.block_rows_hint_for(8, 64, 2, dspark.COMPACT) == 4    # G = 32: 128 columns
    assert dspark.block_rows_hint_for(8, 128, 2, dspark.COMPACT) == 9   # G = 64: whole block
    assert bench.query_tile(W.WORKLOADS["mla"], 9) == "mla"


def test_source_hash_keys_code_not_comments(tmp_path):
    """A committed traffic figure stays valid through a comment or layout edit of its
    sources and is dropped by any change of code."""
    a = tmp_path / "k.cu"
    a.write_text("int f(int x) {\n  return x + 1;  // one\n}\n/* note */\n")
    h0 = bench.src_hash([str(a)])
    a.write_text("// header\nint f(int x)\n{\n    return x + 1;  // other words\n}\n")
    assert bench.src_hash([str(a)]) == h0
    a.write_text("int f(int x) {\n  return x + 2;\n}\n")
    assert bench.src_hash([str(a)]) != h0


def test_oracle_baseline_complete_steps_one_core_and_pool():
    """The CPU baseline times complete oracle steps; the pooled run (spawned worker
    processes over memory-mapped inputs) computes what the one-core run computes."""
    from oracle import dspark_oracle as O
    inp = W.make_inputs(W.WORKLOADS["tiny"], 1)
    ob = bench.OracleBaseline(inp, O.COMPACT, cores=2)
    try:
        h = ob.h
        sch = O.schedule(h["conf"], h["conf_is_logit"], h["sts_temp"], h["cost_table"],
                         ob.wl.max_tokens, O.COMPACT)
        pk = O.pack(sch.windows, h["ctx_len"], h["anchor"], h["draft_tok"], h["tiers"],
                    O.COMPACT, ob.wl.gamma)
        tasks = [(r, int(pk.cu_seqlens[r]), int(pk.cu_seqlens[r + 1]), int(sch.windows[r]))
                 for r in range(ob.wl.B)]
        one = [bench._oracle_request(t) for t in tasks]
        many = sorted(ob.start_pool().map(bench._oracle_request, tasks))
        assert one == many
        assert ob.step(False) > 0 and ob.step(True) > 0
    finally:
        ob.close()
    assert not os.path.exists(ob.folder)

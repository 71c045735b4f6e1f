"""dspark_accept_noalloc (fixed library scratch) against dspark_accept (caller
workspace): identical outputs on two consecutive calls.  GPU only; collected last
so that it runs both after the other tests and alone in a fresh process."""
import pytest
import torch

import harness
import workloads as W
from oracle import dspark_oracle as O

pytestmark = pytest.mark.gpu


def _outputs(B, gamma, dev):
    i32 = dict(dtype=torch.int32, device=dev)
    return {
        "accept_len": torch.full((B,), -7, **i32),
        "cap_len": torch.full((B,), -7, **i32),
        "out_tok": torch.full((B,), -7, **i32),
        "cstar": torch.full((B, gamma), 3.0, dtype=torch.float32, device=dev),
        "fallback": torch.full((B,), -7, **i32),
    }


def _same(a, b):
    for k in a:
        torch.testing.assert_close(a[k], b[k], rtol=0, atol=0, equal_nan=True, msg=k)


@pytest.mark.parametrize("wl_name,mode", [("tiny", O.COMPACT), ("qwen3_8b", O.CAP_ACCEPT),
                                          ("mixed256", O.STATIC)])
def test_noalloc_matches_workspace_call(wl_name, mode):
    import speculative_decoding_verification_dspark_gb300 as dspark
    wl = W.WORKLOADS[wl_name]
    inp = W.make_inputs(wl, 3, device=W.gen_device(wl))
    d, step = harness.prepare(inp, mode)
    dev = step.cu_seqlens.device
    dspark.read_device_error()

    # Fill the shared scratch with an unrelated problem first (another workload,
    # mode and shape), so that a stale entry the compared calls failed to rewrite
    # would show up as a difference.
    other = W.WORKLOADS["mixed256"].replace(name="noalloc_fill", B=96, ctx=("const", 32),
                                             vocab=65536, p_dtype="f32")
    oin = W.make_inputs(other, 7, device=W.gen_device(other))
    od, ostep = harness.prepare(oin, O.STATIC)
    junk = _outputs(other.B, other.gamma, dev)
    dspark.accept_noalloc(od["p_target"], od["p_draft"], od["draft_tok"], od["uniforms"],
                          od["exp_noise"], ostep.windows, ostep.cu_seqlens, O.STATIC,
                          junk["accept_len"], junk["cap_len"], junk["out_tok"], junk["cstar"],
                          junk["fallback"])
    torch.cuda.synchronize()
    del od, ostep, oin, junk
    ref = _outputs(wl.B, wl.gamma, dev)
    dspark.accept(d["p_target"], d["p_draft"], d["draft_tok"], d["uniforms"], d["exp_noise"],
                  step.windows, step.cu_seqlens, mode, ref["accept_len"], ref["cap_len"],
                  ref["out_tok"], ref["cstar"], ref["fallback"], step.ws_accept)
    runs = []
    for _ in range(2):  # consecutive calls share the one scratch array
        got = _outputs(wl.B, wl.gamma, dev)
        dspark.accept_noalloc(d["p_target"], d["p_draft"], d["draft_tok"], d["uniforms"],
                              d["exp_noise"], step.windows, step.cu_seqlens, mode,
                              got["accept_len"], got["cap_len"], got["out_tok"], got["cstar"],
                              got["fallback"])
        runs.append(got)
    torch.cuda.synchronize()
    assert dspark.read_device_error() == 0
    _same(ref, runs[0])
    _same(ref, runs[1])


def test_noalloc_rejects_oversized_problem():
    """A problem whose scratch would exceed the fixed array is refused on the host
    (DSPARK_ENOSPACE) and nothing is launched: the size check reads only the sizes,
    so the row count is passed directly with small buffers behind it."""
    import ctypes
    import speculative_decoding_verification_dspark_gb300 as dspark
    wl = W.WORKLOADS["tiny"]
    dev = torch.device("cuda")
    B, gamma, V = wl.B, wl.gamma, 151936
    rows = 16384  # 16384 rows x 19 chunks x 32 B > the fixed scratch
    p_t = torch.zeros(8, V, dtype=torch.bfloat16, device=dev)
    p_d = torch.zeros(B, gamma, V, dtype=torch.bfloat16, device=dev)
    noise = torch.ones(B, V, dtype=torch.float32, device=dev)
    i32 = dict(dtype=torch.int32, device=dev)
    draft, win, cu = (torch.zeros(B, gamma, **i32), torch.zeros(B, **i32),
                      torch.zeros(B + 1, **i32))
    u = torch.full((B, gamma), 0.5, device=dev)
    out = _outputs(B, gamma, dev)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = dspark.lib().dspark_accept_noalloc(
        P(p_t), P(p_d), dspark.BF16, V, P(draft), P(u), P(noise), P(win), P(cu), O.COMPACT, B,
        gamma, rows, P(out["accept_len"]), P(out["cap_len"]), P(out["out_tok"]), P(out["cstar"]),
        P(out["fallback"]), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == -4  # DSPARK_ENOSPACE
    torch.cuda.synchronize()
    assert int(out["accept_len"][0]) == -7  # nothing was launched

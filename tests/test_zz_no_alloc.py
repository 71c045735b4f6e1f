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
    import speculative_decoding_verification_dspark_gb300 as dspark
    wl = W.WORKLOADS["tiny"]
    dev = torch.device("cuda")
    B, gamma, V = wl.B, wl.gamma, 151936
    rows = 16384  # 16384 rows x 19 chunks x 32 B > the fixed scratch
    # contents unused: the size check runs on the host before anything is read
    p_t = torch.empty(rows, V, dtype=torch.bfloat16, device=dev)
    p_d = torch.empty(B, gamma, V, dtype=torch.bfloat16, device=dev)
    noise = torch.ones(B, V, dtype=torch.float32, device=dev)
    i32 = dict(dtype=torch.int32, device=dev)
    out = _outputs(B, gamma, dev)
    with pytest.raises(dspark.DSparkError):
        dspark.accept_noalloc(p_t, p_d, torch.zeros(B, gamma, **i32),
                              torch.full((B, gamma), 0.5, device=dev), noise,
                              torch.zeros(B, **i32), torch.zeros(B + 1, **i32), O.COMPACT,
                              out["accept_len"], out["cap_len"], out["out_tok"], out["cstar"],
                              out["fallback"])
    assert int(out["accept_len"][0]) == -7  # nothing was launched

"""GPU parity of the block-accept estimate (dspark_block_accept_estimate): bit-exact
against the oracle on the step's own acceptance outputs, and, against a cap-accept
run of the same inputs, every interval holds the full-block cap and every exact
value equals it."""
import numpy as np
import pytest
import torch

import harness
import workloads as W
from oracle import dspark_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    import __graft_entry__ as g
    g.build()
    import speculative_decoding_verification_dspark_gb300 as p
    return p


def _run(pkg, inp, mode):
    d, step = harness.prepare(inp, mode)
    step.run(d, mode)
    lo, hi = pkg.block_accept_estimate(d["p_target"], d["p_draft"], d["draft_tok"], d["uniforms"],
                                       step.windows, step.cu_seqlens, mode, step.accept_len,
                                       step.cap_len)
    torch.cuda.synchronize()
    assert pkg.read_device_error() == 0
    cpu = lambda t: t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()
    return {"lo": lo.cpu().numpy(), "hi": hi.cpu().numpy(), "windows": step.windows.cpu().numpy(),
            "cu": step.cu_seqlens.cpu().numpy(), "L": step.accept_len.cpu().numpy(),
            "cap": step.cap_len.cpu().numpy(), "p_target": cpu(d["p_target"]),
            "p_draft": cpu(d["p_draft"]), "draft_tok": d["draft_tok"].cpu().numpy(),
            "uniforms": d["uniforms"].cpu().numpy()}


CASES = [("tiny", "f32", 0), ("tiny", "bf16", 1), ("qwen3_8b", "f32", 0)]


@pytest.mark.parametrize("name,pdt,seed", CASES)
def test_block_accept_estimate_matches_oracle_and_brackets_cap_accept(pkg, name, pdt, seed):
    wl = W.WORKLOADS[name].replace(p_dtype=pdt)
    gamma = wl.gamma
    inp = W.make_inputs(wl, seed, device=W.gen_device(wl))
    c = _run(pkg, inp, W.MODE_COMPACT)
    lo, hi = O.block_accept_estimate(c["p_target"], c["p_draft"], c["draft_tok"], c["uniforms"],
                                     c["windows"], c["cu"], c["L"], c["cap"], O.COMPACT, gamma)
    assert np.array_equal(c["lo"], lo) and np.array_equal(c["hi"], hi)
    f = _run(pkg, inp, W.MODE_CAP_ACCEPT)
    assert np.array_equal(f["windows"], c["windows"])
    cap = f["cap"]
    assert np.all(c["lo"] <= cap) and np.all(cap <= c["hi"])
    exact = c["lo"] == c["hi"]
    assert np.array_equal(c["lo"][exact], cap[exact])
    # the other modes report the cap they verified
    assert np.array_equal(f["lo"], cap) and np.array_equal(f["hi"], cap)

"""Failure detection without a GPU fault: the acceptance pass's producer waits on a
barrier nothing arrives at (the wait probe) with a 50 us limit; the wait runs out,
the kernel reports DSPARK_DEVERR_WAIT_TIMEOUT and every role stops with nothing left
in flight (the context intact); the next call, probe off and default limit, gives the
outputs of a normal call."""
import pytest
import torch

import harness
import workloads as W
from oracle import dspark_oracle as O

pytestmark = pytest.mark.gpu


def _outs(step):
    return [step.accept_len.clone(), step.cap_len.clone(), step.out_tok.clone(),
            step.cstar.clone(), step.fallback.clone()]


def _same_bits(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


@pytest.mark.parametrize("mode", [O.COMPACT, O.CAP_ACCEPT])
def test_accept_wait_timeout_is_reported_and_the_next_call_is_correct(mode):
    import __graft_entry__ as g
    g.build()
    import speculative_decoding_verification_dspark_gb300 as dspark
    wl = W.WORKLOADS["qwen3_8b"]
    inp = W.make_inputs(wl, 5, device=W.gen_device(wl))
    d, step = harness.prepare(inp, mode)
    dspark.read_device_error()
    step.accept(d, mode)
    torch.cuda.synchronize()
    assert dspark.read_device_error() == 0
    ref = _outs(step)
    try:
        # a wait on a barrier nothing arrives at, limited to 50 us
        dspark.set_wait_limit_ns(50_000)
        dspark.set_wait_probe(True)
        step.accept(d, mode)
        torch.cuda.synchronize()
        err = dspark.read_device_error()
    finally:
        dspark.set_wait_probe(False)
        dspark.set_wait_limit_ns(0)
    assert err & 0x8, f"device error word {err:#x}"
    for t in (step.accept_len, step.cap_len, step.out_tok, step.cstar, step.fallback):
        t.fill_(-3)   # the recovery call must write every output
    step.accept(d, mode)
    torch.cuda.synchronize()
    assert dspark.read_device_error() == 0
    for a, b in zip(ref, _outs(step)):
        assert _same_bits(a, b)

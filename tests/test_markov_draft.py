"""GPU parity of the Markov-head draft sampler (dspark_markov_draft) against the
oracle, on seeded inputs of the draft workloads.

Tolerances come from the arithmetic.  A logit is U + sum_j W1[x, j] W2[j, v]: the
bf16 products are exact in fp32, and the fp32 accumulation of 257 terms errs by at
most 258 * 2^-24 * (sum_j |W1[x, j] W2[j, v]| + |U|) = delta (the standard bound of
recursive summation, whatever the order).  The kernel's exp2 / log2 approximations
and the conversions to the log2 domain add less than 1e-5 in the natural-log domain.
So ln p_gpu is within 2 delta + 1e-5 of ln p (the logit, the row's max and its log
sum each move by at most delta), and the race key ln(p / e) of every entry within
delta + 1e-5: the token the kernel picks has an exact key within 2 (delta + 1e-5)
of the maximum.  A token is checked as equal to the oracle's, or as such a near
tie; every position is checked on the kernel's own prefix (the oracle conditions
on the kernel's tokens)."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import dspark_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    import __graft_entry__ as g
    g.build()
    import speculative_decoding_verification_dspark_gb300 as p
    return p


def _run(pkg, inp, sampler=None):
    V = inp["U"].shape[2]
    sampler = sampler or pkg.MarkovDraft(V)
    tok, p = sampler(inp["U"], inp["W1"], inp["W2"], inp["anchor"], inp["exp_noise"])
    torch.cuda.synchronize()
    assert pkg.read_device_error() == 0
    return tok.cpu().numpy(), p.cpu().numpy(), sampler


def _delta(U, aW1, aW2, prev):
    """258 * 2^-24 * (|W1[prev]| @ |W2| + |U|), per entry: the accumulation bound."""
    return 258.0 * 2.0 ** -24 * (aW1[prev] @ aW2 + np.abs(U))


def _check_rows(inp, tok, p, rows):
    U = inp["U"].cpu().numpy()[rows].astype(np.float64)
    W1 = inp["W1"].float().cpu().numpy().astype(np.float64)
    W2 = inp["W2"].float().cpu().numpy().astype(np.float64)
    e = inp["exp_noise"].cpu().numpy()[rows]
    anchor = inp["anchor"].cpu().numpy()[rows]
    g_tok = tok[rows]
    o_tok, o_p, o_k = O.markov_draft(U, W1, W2, anchor, e, tokens_given=g_tok)
    gamma = U.shape[1]
    aW1, aW2 = np.abs(W1), np.abs(W2)
    n_tie = 0
    for i in range(len(rows)):
        for k in range(gamma):
            prev = int(anchor[i]) if k == 0 else int(g_tok[i, k - 1])
            d = _delta(U[i, k], aW1, aW2, prev).max()
            tol_ln = 2 * d + 1e-5
            pg = p[rows[i], k].astype(np.float64)
            po = o_p[i, k]
            bad = np.abs(pg - po) > po * np.expm1(tol_ln) + 1e-30
            assert not bad.any(), (rows[i], k, int(np.argmax(bad)), pg[bad][:3], po[bad][:3], tol_ln)
            gt, ot = int(g_tok[i, k]), int(o_tok[i, k])
            assert 0 <= gt < U.shape[2]
            if gt != ot:
                gap = np.log(o_k[i, k, ot]) - np.log(o_k[i, k, gt])
                assert gap <= 2 * (d + 1e-5), (rows[i], k, gt, ot, gap, d)
                n_tie += 1
    return n_tie


@pytest.mark.parametrize("name", ["markov_one", "markov_small", "markov_g32", "markov_ragged",
                                  "markov_wide"])
def test_markov_draft_matches_the_oracle(pkg, name):
    cfg = W.MARKOV_WORKLOADS[name]
    inp = W.make_markov_inputs(cfg["B"], cfg["gamma"], cfg["V"], seed=3, device="cuda")
    tok, p, _ = _run(pkg, inp)
    n_tie = _check_rows(inp, tok, p, np.arange(cfg["B"]))
    # near ties are rare on continuous draws
    assert n_tie <= max(1, cfg["B"] * cfg["gamma"] // 50)


def test_markov_draft_full_vocabulary_sampled_rows(pkg):
    """Qwen3-8B vocabulary at the full batch and block (the timed configuration):
    every row's p sums to 1; eight sampled rows against the oracle."""
    cfg = W.MARKOV_WORKLOADS["markov_qwen3_8b"]
    inp = W.make_markov_inputs(cfg["B"], cfg["gamma"], cfg["V"], seed=0, device="cuda")
    tok, p, _ = _run(pkg, inp)
    s = p.astype(np.float64).sum(axis=2)
    assert np.all(np.abs(s - 1.0) < 1e-4)
    rows = np.random.default_rng(7).choice(cfg["B"], 8, replace=False)
    n_tie = _check_rows(inp, tok, p, np.sort(rows))
    assert n_tie <= 1


def test_markov_draft_repeats_exactly_and_leaves_its_workspace_ready(pkg):
    """Two calls on one workspace give identical tokens and probabilities, and the
    grid-barrier word is back to zero in its low 31 bits after each."""
    cfg = W.MARKOV_WORKLOADS["markov_ragged"]
    inp = W.make_markov_inputs(cfg["B"], cfg["gamma"], cfg["V"], seed=5, device="cuda")
    tok1, p1, sampler = _run(pkg, inp)
    word = sampler.ws[:4].view(torch.int32).item() & 0x7FFFFFFF
    assert word == 0
    tok2, p2, _ = _run(pkg, inp, sampler)
    assert np.array_equal(tok1, tok2)
    assert np.array_equal(p1.view(np.int32), p2.view(np.int32))
    assert (sampler.ws[:4].view(torch.int32).item() & 0x7FFFFFFF) == 0

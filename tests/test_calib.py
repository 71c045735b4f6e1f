"""Calibration tooling on the GPU against the oracle: the labelled samples the
step's outcomes give (collected step after step on the device), the ECE of the
calibrated survival, and the STS temperature refit."""
import numpy as np
import pytest
import torch

import harness
import workloads as W
from oracle import dspark_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _npy(t):
    return t.detach().cpu().numpy()


def _merge(acc, new):
    for j, pos in enumerate(new):
        acc[j].extend(pos)
    return acc


@pytest.mark.parametrize("mode", ["compact", "cap_accept"])
def test_collect_from_steps_matches_oracle(mode):
    """Four tiny steps: the device store equals the oracle's samples of the same
    steps (positions, order, labels; survival and a_hat to one fp32 ulp), and the
    ECE and refit of the store equal the oracle's on its own samples."""
    import speculative_decoding_verification_dspark_gb300 as dspark
    m = W.MODE_NAMES[mode]
    wl = W.WORKLOADS["tiny"]
    store = dspark.CalibStore(wl.gamma, 64)
    oracle_samples = [[] for _ in range(wl.gamma)]
    for seed in range(4):
        inp = W.make_inputs(wl, 10 + seed)
        d, step = harness.prepare(inp, m)
        step.run(d, m)
        store.collect(step.survival, step.a_hat, step.windows, step.cap_len, m)
        torch.cuda.synchronize()
        assert dspark.read_device_error() == 0
        # the oracle's own step (schedule, pack, accept) on the same inputs
        npi = {k: (v.float().numpy() if v.dtype == torch.bfloat16 else v.numpy())
               for k, v in inp.items() if isinstance(v, torch.Tensor)}
        c = O.confidence(npi["conf"], inp["conf_is_logit"])
        a = O.prefix_survival(c)
        sch = O.schedule(npi["conf"], inp["conf_is_logit"], npi["sts_temp"], npi["cost_table"],
                         wl.max_tokens, m)
        assert not sch.listed
        pk = O.pack(sch.windows, npi["ctx_len"], npi["anchor"], npi["draft_tok"], npi["tiers"],
                    m, wl.gamma)
        pt = W.to_packed(inp["p_target_dense"], torch.as_tensor(pk.cu_seqlens), pk.tier).numpy()
        acc = O.accept(pt[:pk.M], npi["p_draft"], npi["draft_tok"], npi["uniforms"],
                       npi["exp_noise"], sch.windows, pk.cu_seqlens, m, wl.gamma)
        _merge(oracle_samples, O.calib_samples(a, sch.a_hat, sch.windows, acc.cap_len, m,
                                               wl.gamma))
    count = _npy(store.count)
    assert count.tolist() == [len(p) for p in oracle_samples]
    for j, pos in enumerate(oracle_samples):
        n = len(pos)
        ga, gh, gy = _npy(store.s_a[j, :n]), _npy(store.s_ahat[j, :n]), _npy(store.s_y[j, :n])
        oa = np.array([x[0] for x in pos], np.float32)
        oh = np.array([x[1] for x in pos], np.float32)
        assert np.array_equal(gy, np.array([x[2] for x in pos], np.int8))
        assert np.all(np.abs(ga.view(np.int32).astype(np.int64) - oa.view(np.int32)) <= 1)
        assert np.all(np.abs(gh.view(np.int32).astype(np.int64) - oh.view(np.int32)) <= 1)
    e, bn, bp, by = store.ece(10)
    oe, ocnt, osp, osy = O.ece(oracle_samples, 10)
    assert _npy(bn).tolist() == ocnt.tolist()
    assert abs(float(e[0]) - oe) < 1e-6
    T = _npy(store.sts_fit(40))
    for j, pos in enumerate(oracle_samples):
        assert abs(float(T[j]) - float(O.sts_fit(pos, 40))) <= 1e-5 * float(T[j]), j


def _synthetic_outcomes(rng, B, gamma, T_true):
    """Requests whose confidence is a running product of c ~ U(0.6, 1), and accept
    outcomes drawn position by position so that P(prefix 1..j accepted) =
    sigmoid(logit(a_j) / T_true): a head that is miscalibrated by T_true."""
    c = rng.uniform(0.6, 1.0, size=(B, gamma)).astype(np.float32)
    a = O.prefix_survival(c)
    z = np.log(a.astype(np.float64)) - np.log1p(-a.astype(np.float64))
    p = 1.0 / (1.0 + np.exp(-z / T_true))
    p = np.minimum.accumulate(p, axis=1)
    cond = p / np.concatenate([np.ones((B, 1)), p[:, :-1]], axis=1)
    u = rng.uniform(0, 1, size=(B, gamma))
    ok = u < cond
    cap = np.where(ok.all(1), gamma, np.argmin(ok, axis=1)).astype(np.int32)
    a_hat = (a * np.float32(0.9)).astype(np.float32)   # any prediction: only binned
    windows = rng.integers(0, gamma + 1, size=B).astype(np.int32)
    return a, a_hat, windows, cap


@pytest.mark.parametrize("mode", ["compact", "cap_accept"])
def test_collect_ece_and_fit_on_many_samples(mode):
    """30 collect calls of 1024 requests (the store overflows in cap-accept mode:
    the first `capacity` samples are kept, count keeps counting); ECE with 15 bins;
    the refit recovers the temperature that generated the labels, and equals the
    oracle's refit of the same samples."""
    import speculative_decoding_verification_dspark_gb300 as dspark
    m = W.MODE_NAMES[mode]
    rng = np.random.default_rng(41)
    B, gamma, cap, T_true = 1024, 8, 20000, 1.6
    store = dspark.CalibStore(gamma, cap)
    samples = [[] for _ in range(gamma)]
    dev = torch.device("cuda")
    for _ in range(30):
        a, ah, w, capl = _synthetic_outcomes(rng, B, gamma, T_true)
        # cap_len as the acceptance reports it: the accepted prefix over the verified
        # positions
        v = np.full(B, gamma, np.int32) if m == O.CAP_ACCEPT else w
        capl = np.minimum(capl, v).astype(np.int32)
        store.collect(torch.from_numpy(a).to(dev), torch.from_numpy(ah).to(dev),
                      torch.from_numpy(w).to(dev), torch.from_numpy(capl).to(dev), m)
        _merge(samples, O.calib_samples(a, ah, w, capl, m, gamma))
    torch.cuda.synchronize()
    assert dspark.read_device_error() == 0
    count = _npy(store.count)
    assert count.tolist() == [len(p) for p in samples]
    kept = [p[:cap] for p in samples]
    for j, pos in enumerate(kept):
        n = len(pos)
        assert np.array_equal(_npy(store.s_a[j, :n]), np.array([x[0] for x in pos], np.float32))
        assert np.array_equal(_npy(store.s_y[j, :n]), np.array([x[2] for x in pos], np.int8))
    e, bn, _, _ = store.ece(15)
    oe, ocnt, _, _ = O.ece(kept, 15)
    assert _npy(bn).tolist() == ocnt.tolist()
    assert abs(float(e[0]) - oe) < 1e-9
    T = _npy(store.sts_fit(36))
    for j in range(gamma):
        To = float(O.sts_fit(kept[j], 36))
        assert abs(float(T[j]) - To) <= 1e-5 * To, (j, T[j], To)
    if m == O.CAP_ACCEPT:   # unbiased labels at every position: the generator's temperature
        assert np.all(np.abs(T - T_true) < 0.15 * T_true), T

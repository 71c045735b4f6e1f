"""Plain CPU oracle for DSpark's confidence-scheduled ragged verification step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code with the CUDA library; the two meet
only through the seeded inputs of ``workloads.py``.

It is written to be read against the pages, not to be fast: plain loops over
requests, rows and draft positions; numpy only for dot products, exp/log and
argmax.  Floating point is fp64 unless the step is an fp32 decision the method
fixes (acceptance test, sampling keys), in which case it is done in fp32 on
exactly-representable inputs.

Sources, cited by short name below:

* [lesson]  "DFlash 到 DSpark in SGLang：解码提速 4.3×，以及 DeepSeek-V4 支持"
            (AI Infra Visualized lesson on DSpark).  Sections "Background",
            "DSpark：sequential head 加验证预算", "Confidence scheduler 与 verify 模式",
            "Ragged verify under full CUDA graphs", "Zero-overhead scheduling 与 kernel".
* [csdn]    DevPress/CSDN article on DSpark in SGLang, sections "2." (verify modes),
            "3." (ragged packing), "4." (additive cost model T(bs,K)), "5." (observability,
            including the block-accept estimator).
* [notes]   "DSpark：投机解码与生产级 Serving 学习笔记", sections "02 · Speculative
            Decoding", "07 · Confidence Head", "08 · Hardware-Aware Prefix Scheduler",
            "09 · End-to-End Cycle".

Parity status per function (what pins it is listed in tests/test_oracle_pins.py):
pinned: confidence sigmoid, survival/STS, greedy schedule, pack, verify
attention (GQA and MLA), acceptance (test, race, fallback, c*), compaction,
calibration samples, ECE and the STS refit, Markov-head draft sampling, the
block-accept estimate.  The composed ``step`` adds no arithmetic of its own and
is pinned only through its parts (no page prints end-to-end values).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

F32 = np.float32
COMPACT, STATIC, CAP_ACCEPT = 0, 1, 2
MARGIN_LIST_REL = 1e-5


# ----------------------------------------------------------------------------
# 1. Confidence, prefix survival, sequential temperature scaling
# ----------------------------------------------------------------------------

def confidence(conf: np.ndarray, is_logit: bool) -> np.ndarray:
    """c_k from the confidence head: a linear layer followed by a sigmoid
    ([notes] §07; [lesson] "DSpark：sequential head 加验证预算").

    The sigmoid is evaluated in fp64 and rounded once to fp32, so c is the
    fp32 number nearest to sigma(z) up to one fp64 rounding (reading A21: the
    pages fix no arithmetic for the scheduler; this one lets two independent
    implementations agree to within one fp32 ulp).
    """
    x = np.asarray(conf, dtype=np.float32)
    if not is_logit:
        return x.copy()
    z = x.astype(np.float64)
    out = np.empty(z.shape, dtype=np.float32)
    for idx in np.ndindex(z.shape):
        out[idx] = F32(1.0 / (1.0 + math.exp(-z[idx]))) if z[idx] > -700 else F32(0.0)
    return out


def prefix_survival(c: np.ndarray) -> np.ndarray:
    """a_j = prod_{i<=j} c_i: position j is only used if positions 1..j all pass,
    so the conditional acceptance probabilities multiply ([notes] §07, the
    survival table; [notes] §15 "为什么 prefix survival probability 要相乘").

    fp32 products taken left to right (each product is one IEEE fp32 rounding).
    """
    B, gamma = c.shape
    a = np.empty((B, gamma), dtype=np.float32)
    for r in range(B):
        acc = F32(c[r, 0])
        a[r, 0] = acc
        for j in range(1, gamma):
            acc = F32(acc * F32(c[r, j]))
            a[r, j] = acc
    return a


def sts_calibrate(a: np.ndarray, temps: np.ndarray) -> np.ndarray:
    """Sequential Temperature Scaling of the cumulative survival ([notes] §07
    "为什么还要做 Sequential Temperature Scaling"; [lesson] "整块连乘是块的存活率，
    STS 再把它校准到真实接受率").

    Reading: a per-position temperature T_j divides the logit of the cumulative
    survival, a_hat_j = sigmoid(logit(a_j) / T_j), computed in fp64 as
    t = (log a - log1p(-a)) / T_j,  a_hat = 1 / (1 + exp(-t)), rounded once to
    fp32.  The result is then clamped to be non-increasing in j (running
    minimum), because a prefix can only survive less as it grows and the
    scheduler must pick prefixes.
    """
    B, gamma = a.shape
    out = np.empty((B, gamma), dtype=np.float32)
    for r in range(B):
        prev = None
        for j in range(gamma):
            x = float(a[r, j])
            if x <= 0.0:
                y = 0.0
            elif x >= 1.0:
                y = 1.0
            else:
                t = (math.log(x) - math.log1p(-x)) / float(temps[j])
                y = 1.0 / (1.0 + math.exp(-t)) if t > -700 else 0.0
            v = F32(y)
            if prev is not None and v > prev:
                v = prev
            out[r, j] = v
            prev = v
    return out


# ----------------------------------------------------------------------------
# 2. Global greedy window scheduler against the step-cost model
# ----------------------------------------------------------------------------

@dataclass
class Schedule:
    windows: np.ndarray            # int32 [B]
    a_hat: np.ndarray              # fp32 [B, gamma] calibrated survival
    M: int                         # B + sum(windows)
    E: float                       # expected committed tokens B + sum of accepted a_hat
    order: list                    # sorted candidates (a_hat, r, j)
    n_accepted: int
    stop_reason: str               # "decline", "budget", "exhausted", "static"
    listed: list = field(default_factory=list)   # near-margin decisions (kind, r, j, rel)


def schedule(conf, conf_is_logit, sts_temp, cost_table, max_tokens, mode) -> Schedule:
    """Per-request verify windows by the global greedy of [notes] §08.3 and
    [lesson] "Confidence scheduler 与 verify 模式".

    All (request, position) candidates are sorted by calibrated survival, high
    to low (ties: request ascending, then position ascending).  Starting from the
    batch itself (E = B expected commits: every request commits at least its
    bonus/correction token; M = B verify rows: one anchor row per request,
    M = bs + K of [csdn] §4), candidates are added one at a time while the
    expected throughput E / T(M) rises strictly, and the walk stops at the first
    candidate that does not raise it, or when M + 1 would exceed the largest
    captured tier.  T is the profiled step-cost table indexed by M.

    Arithmetic (reading A21): E is kept in fp64 and the two ratios are compared
    cross-multiplied in fp64 (T > 0).  Here E is summed in sorted order; any other
    order gives the same decisions outside the listing margin, because an fp64
    sum of n <= 4096 terms in [0, 1] is within n * 2^-53 * E of exact (below
    1e-12 relative), whereas an fp32 running sum could be off by n * 2^-24
    (2.4e-4 at n = 4096), more than the margin.  Every decision whose relative
    margin |lhs - rhs| / rhs is below 1e-5 is recorded in ``listed``; so are the
    requests of all candidates within 1e-5 (relative) of the stopping
    candidate's survival when they belong to two or more requests, since a
    rounding of a_hat could reorder them across the stop.

    static mode verifies the whole block: w_r = gamma.
    """
    c = confidence(conf, conf_is_logit)
    a = prefix_survival(c)
    ah = sts_calibrate(a, np.asarray(sts_temp, dtype=np.float32))
    B, gamma = ah.shape
    cost = np.asarray(cost_table, dtype=np.float32)
    windows = np.zeros(B, dtype=np.int32)
    if mode == STATIC:
        E = float(B) + sum(float(ah[r, j]) for r in range(B) for j in range(gamma))
        windows[:] = gamma
        return Schedule(windows, ah, B * (gamma + 1), E, [], B * gamma, "static")
    cands = [(float(ah[r, j]), r, j) for r in range(B) for j in range(gamma)]
    cands.sort(key=lambda t: (-t[0], t[1], t[2]))
    E, M = float(B), B
    listed = []
    stop = "exhausted"
    k = 0
    for k, (v, r, j) in enumerate(cands):
        if M + 1 > max_tokens:
            stop = "budget"
            break
        # throughput rises iff (E + v) / T[M+1] > E / T[M]; with T > 0 this is
        # (E + v) * T[M] > E * T[M+1], evaluated in fp64 without a division
        lhs = (E + v) * float(cost[M])
        rhs = E * float(cost[M + 1])
        rel = abs(lhs - rhs) / rhs
        if lhs > rhs:
            if rel < MARGIN_LIST_REL:
                listed.append(("accept", r, j, rel))
            assert windows[r] == j, "candidates of one request must arrive in position order"
            E += v
            M += 1
            windows[r] += 1
        else:
            if rel < MARGIN_LIST_REL:
                listed.append(("stop", r, j, rel))
            stop = "decline"
            break
    else:
        k = len(cands)
    n_acc = int(windows.sum())
    if stop in ("decline", "budget") and n_acc < len(cands):
        # candidates whose survival is within the margin of the stopping one: a
        # one-ulp difference in a_hat could put any of them on either side
        v_stop = cands[n_acc][0]
        band = [(k2, v2, r2, j2) for k2, (v2, r2, j2) in enumerate(cands)
                if abs(v2 - v_stop) <= MARGIN_LIST_REL * v_stop]
        if len({r2 for (_, _, r2, _) in band}) > 1 and v_stop > 0:
            for (k2, v2, r2, j2) in band:
                listed.append(("tie", r2, j2, abs(v2 - v_stop) / v_stop))
    return Schedule(windows, ah, M, E, cands, n_acc, stop, listed)


# ----------------------------------------------------------------------------
# 3. Head-to-tail packing and tier selection
# ----------------------------------------------------------------------------

@dataclass
class Pack:
    cu_seqlens: np.ndarray   # int32 [B+1]
    M: int
    tier: int
    row_req: np.ndarray      # int32 [tier]   (-1 on padding rows)
    row_pos: np.ndarray      # int32 [tier]   absolute position ctx_r + i (-1 on padding)
    row_tok: np.ndarray      # int32 [tier]   anchor for i = 0, d_i for i >= 1 (-1 on padding)


def verify_lengths(windows, mode, gamma) -> np.ndarray:
    """Draft positions each request sends to the target: the window in compact
    mode, the whole block in static and cap-accept mode ([lesson] "Confidence
    scheduler 与 verify 模式"; [csdn] §2)."""
    w = np.asarray(windows, dtype=np.int64)
    if mode == CAP_ACCEPT:
        return np.full_like(w, gamma)
    return w


def pack(windows, ctx_len, anchor, draft_tok, tiers, mode, gamma) -> Pack:
    """Head-to-tail packing with cu_seqlens and tier rounding ([lesson] "Ragged
    verify under full CUDA graphs"; [csdn] §3).

    Request r occupies n_r = 1 + (verified drafts) consecutive rows: the anchor
    (the previous bonus/correction token) and the drafts d_1..d_n.  cu_seqlens
    is the exclusive prefix sum of n_r.  The tier is the smallest captured tier
    >= M; if M exceeds every tier the step runs unpadded (tier = M).
    """
    B = len(windows)
    nver = verify_lengths(windows, mode, gamma)
    n = 1 + nver
    cu = np.zeros(B + 1, dtype=np.int64)
    for r in range(B):
        cu[r + 1] = cu[r] + n[r]
    M = int(cu[B])
    tier = M
    for t in sorted(int(x) for x in tiers):
        if t >= M:
            tier = t
            break
    row_req = np.full(tier, -1, dtype=np.int32)
    row_pos = np.full(tier, -1, dtype=np.int32)
    row_tok = np.full(tier, -1, dtype=np.int32)
    for r in range(B):
        for i in range(int(n[r])):
            row = int(cu[r]) + i
            row_req[row] = r
            row_pos[row] = int(ctx_len[r]) + i
            row_tok[row] = int(anchor[r]) if i == 0 else int(draft_tok[r, i - 1])
    return Pack(cu.astype(np.int32), M, tier, row_req, row_pos, row_tok)


# ----------------------------------------------------------------------------
# 4. Varlen verify attention over the paged KV cache
# ----------------------------------------------------------------------------

def _cached_rows(cache, page_table_row, ctx, page_size):
    """Rows 0..ctx-1 of one request's paged cache, in position order."""
    rows = []
    for p in range(ctx):
        page = int(page_table_row[p // page_size])
        rows.append(cache[page, p % page_size])
    if not rows:
        return np.zeros((0,) + cache.shape[2:], dtype=np.float64)
    return np.stack(rows).astype(np.float64)


def verify_attention_gqa(q, k_new, v_new, k_cache, v_cache, page_table, ctx_len, cu_seqlens,
                         Hq, Hkv, scale):
    """Verify attention of the packed rows ([lesson] "Ragged verify under full
    CUDA graphs"; [csdn] §3): every packed row attends only to its own request's
    keys -- the committed context (paged) and the block rows up to and including
    itself (causal within the block).

    Definition, fp64: for row (r, i) and query head h (KV head h // (Hq/Hkv)),
    s_k = scale * <q, k_k> over keys k = cache[0..ctx_r) ++ block[0..i],
    o = sum_k softmax(s)_k v_k, lse = log sum_k exp(s_k).

    q [rows, Hq, D], k_new/v_new [rows, Hkv, D], caches [pages, P, Hkv, D].
    Returns o [M, Hq, Dv] and lse [M, Hq] for the M packed rows.
    """
    q = np.asarray(q, dtype=np.float64)
    kn = np.asarray(k_new, dtype=np.float64)
    vn = np.asarray(v_new, dtype=np.float64)
    B = len(ctx_len)
    P = k_cache.shape[1]
    G = Hq // Hkv
    M = int(cu_seqlens[B])
    o = np.zeros((M, Hq, vn.shape[-1]), dtype=np.float64)
    lse = np.zeros((M, Hq), dtype=np.float64)
    for r in range(B):
        c0, c1 = int(cu_seqlens[r]), int(cu_seqlens[r + 1])
        kc = _cached_rows(k_cache, page_table[r], int(ctx_len[r]), P)
        vc = _cached_rows(v_cache, page_table[r], int(ctx_len[r]), P)
        for i in range(c1 - c0):
            keys = np.concatenate([kc, kn[c0:c0 + i + 1]], axis=0)     # [Nk, Hkv, D]
            vals = np.concatenate([vc, vn[c0:c0 + i + 1]], axis=0)
            for h in range(Hq):
                kv = h // G
                s = scale * (keys[:, kv, :] @ q[c0 + i, h])
                m = s.max()
                e = np.exp(s - m)
                l = e.sum()
                o[c0 + i, h] = (e @ vals[:, kv, :]) / l
                lse[c0 + i, h] = m + math.log(l)
    return o, lse


def verify_attention_mla(q, latent_new, latent_cache, page_table, ctx_len, cu_seqlens, d_v, scale):
    """MLA-shaped verify attention (the latent-KV path the lesson's "Ragged
    verify under full CUDA graphs" names for DeepSeek-V4): all query heads share
    one latent vector per token; keys are the full latent (qk dim), values its
    first d_v components.  Same causal-within-block key set as the GQA case.

    q [rows, H, Dqk], latent_new [rows, Dqk], latent_cache [pages, P, Dqk].
    """
    q = np.asarray(q, dtype=np.float64)
    ln = np.asarray(latent_new, dtype=np.float64)
    B = len(ctx_len)
    P = latent_cache.shape[1]
    H = q.shape[1]
    M = int(cu_seqlens[B])
    o = np.zeros((M, H, d_v), dtype=np.float64)
    lse = np.zeros((M, H), dtype=np.float64)
    for r in range(B):
        c0, c1 = int(cu_seqlens[r]), int(cu_seqlens[r + 1])
        lc = _cached_rows(latent_cache, page_table[r], int(ctx_len[r]), P)
        for i in range(c1 - c0):
            keys = np.concatenate([lc, ln[c0:c0 + i + 1]], axis=0)     # [Nk, Dqk]
            s = scale * (q[c0 + i] @ keys.T)                             # [H, Nk]
            m = s.max(axis=1, keepdims=True)
            e = np.exp(s - m)
            l = e.sum(axis=1, keepdims=True)
            o[c0 + i] = (e @ keys[:, :d_v]) / l
            lse[c0 + i] = (m + np.log(l))[:, 0]
    return o, lse


# ----------------------------------------------------------------------------
# 5. Prefix speculative-sampling acceptance, bonus/correction token, c* label
# ----------------------------------------------------------------------------

@dataclass
class Accept:
    accept_len: np.ndarray   # int32 [B]  committed drafts
    cap_len: np.ndarray      # int32 [B]  accepted prefix over the verified positions
    out_tok: np.ndarray      # int32 [B]  bonus (window fully accepted) or correction token
    cstar: np.ndarray        # fp32 [B, gamma], NaN where no target row exists
    residual_fallback: np.ndarray   # bool [B] all-zero residual, sampled from p_t instead


def _race_argmax(weights_f32: np.ndarray, exp_noise_f32: np.ndarray) -> tuple:
    """Gumbel-max in its exponential-race form: argmax_v w_v / e_v, e_v ~ Exp(1).

    argmax log w_v + G_v with G_v = -log e_v is the same index (reading A11 of
    the Gumbel-max draw in [lesson] "Background" and [notes] §02).  Keys are fp32
    quotients; the lowest index wins ties.  An entry whose weight is not positive
    (zero, or NaN) has log w = -inf and never wins, whatever its noise; a key that
    is NaN never wins either.  If no weight is positive the draw is undefined and
    the lowest index (0) is returned.  Returns (index, best key, any positive
    weight).
    """
    w = np.asarray(weights_f32, dtype=np.float32)
    e = np.asarray(exp_noise_f32, dtype=np.float32)
    live = w > 0
    if not np.any(live):
        return 0, float("-inf"), False
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        q = (w / e).astype(np.float32)
    keys = np.where(live & ~np.isnan(q), q, np.float32(-np.inf))
    idx = int(np.argmax(keys))
    return idx, float(keys[idx]), True


def accept(p_target, p_draft, draft_tok, uniforms, exp_noise, windows, cu_seqlens, mode, gamma) -> Accept:
    """Prefix speculative sampling ([notes] §02 "接受是前缀式的", [lesson]
    "Background", [lesson] "Confidence scheduler 与 verify 模式").

    p_target [rows, V]: packed verify rows; row cu_seqlens[r] + i is the target
    distribution for in-block position i + 1.  p_draft [B, gamma, V] is the
    drafter's distribution for positions 1..gamma.

    * Test, fp32: draft d_j is accepted iff u_j * p_d(d_j) <= p_t(d_j); the
      accepted prefix ends at the first rejection (later drafts are discarded).
    * compact / static: the test runs over the verified positions 1..w_r.
      cap-accept: it runs over the whole block (-> cap_len), and the commit is
      min(cap, w_r), which is exactly what compact commits.
    * Token: after a rejection at position L+1 <= w_r, a correction drawn from
      the residual max(0, p_t - p_d) at that position; when the whole window is
      accepted, a bonus drawn from p_t at position w_r + 1 (the bonus is the
      same token in every mode).  Draws are the exponential race against the
      per-request Exp(1) noise row; entries of zero weight never win.  A
      residual with no positive entry (reachable only through rounding) falls
      back to p_t at that position.
    * c*_j = 1 - 1/2 ||p_d,j - p_t,j||_1 ([notes] §07 training label) for every
      position j <= gamma that has a target row: j <= w_r + 1 in compact mode,
      j <= gamma otherwise.  fp64 sum, rounded to fp32.
    """
    B = len(windows)
    V = p_target.shape[1]
    L_out = np.zeros(B, dtype=np.int32)
    cap_out = np.zeros(B, dtype=np.int32)
    tok_out = np.zeros(B, dtype=np.int32)
    fb = np.zeros(B, dtype=bool)
    cstar = np.full((B, gamma), np.nan, dtype=np.float32)
    for r in range(B):
        w = int(windows[r])
        base = int(cu_seqlens[r])
        test_len = gamma if mode == CAP_ACCEPT else w
        L = 0
        for j in range(1, test_len + 1):
            x = int(draft_tok[r, j - 1])
            pt = F32(p_target[base + j - 1, x])
            pd = F32(p_draft[r, j - 1, x])
            if F32(F32(uniforms[r, j - 1]) * pd) <= pt:
                L += 1
            else:
                break
        cap = L
        commit = min(L, w)
        noise = np.asarray(exp_noise[r], dtype=np.float32)
        if commit < w:
            row_t = np.asarray(p_target[base + commit], dtype=np.float32)
            row_d = np.asarray(p_draft[r, commit], dtype=np.float32)
            resid = np.maximum(F32(0), (row_t - row_d).astype(np.float32))
            tok, _, any_pos = _race_argmax(resid, noise)
            if not any_pos:  # no positive residual entry (reading A12)
                fb[r] = True
                tok, _, _ = _race_argmax(row_t, noise)
        else:
            row_t = np.asarray(p_target[base + w], dtype=np.float32)
            tok, _, _ = _race_argmax(row_t, noise)
        n_rows = int(cu_seqlens[r + 1]) - base
        for j in range(1, min(n_rows, gamma) + 1):
            d = np.asarray(p_draft[r, j - 1], dtype=np.float64)
            t = np.asarray(p_target[base + j - 1], dtype=np.float64)
            cstar[r, j - 1] = F32(1.0 - 0.5 * np.abs(d - t).sum())
        L_out[r], cap_out[r], tok_out[r] = commit, cap, tok
    return Accept(L_out, cap_out, tok_out, cstar, fb)


# ----------------------------------------------------------------------------
# 6. Compact scatter of accepted KV rows and page-table append
# ----------------------------------------------------------------------------

@dataclass
class Compact:
    page_table: np.ndarray
    ctx_len: np.ndarray
    anchor: np.ndarray
    free_top: int
    committed: np.ndarray      # int32 [B, gamma+1], -1 past n_committed
    n_committed: np.ndarray    # int32 [B]
    k_cache: np.ndarray
    v_cache: np.ndarray | None


class NoSpace(Exception):
    pass


def compact(k_new, v_new, cu_seqlens, accept_len, out_tok, draft_tok, page_size,
            page_table, ctx_len, anchor, free_pages, free_top, k_cache, v_cache) -> Compact:
    """Commit the step ([lesson] "Zero-overhead scheduling 与 kernel": compact
    scatter and a device-resident page table; [notes] §09 "进入下一轮").

    For each request in order: the anchor row and the accepted draft rows
    (rows 0..L_r of its segment) are written to cache positions ctx_r..ctx_r+L_r;
    new pages are popped from the top of the free-page stack as positions cross
    page boundaries and appended to the request's page-table row; ctx_r grows by
    L_r + 1; the bonus/correction token becomes the next anchor; the committed
    tokens are d_1..d_L followed by that token.  Rejected rows are never written.
    """
    pt = np.array(page_table, dtype=np.int32, copy=True)
    ctx = np.array(ctx_len, dtype=np.int32, copy=True)
    anc = np.array(anchor, dtype=np.int32, copy=True)
    kc = np.array(k_cache, copy=True)
    vc = None if v_cache is None else np.array(v_cache, copy=True)
    top = int(free_top)
    B = len(ctx)
    gamma = draft_tok.shape[1]
    P = page_size
    committed = np.full((B, gamma + 1), -1, dtype=np.int32)
    ncom = np.zeros(B, dtype=np.int32)
    for r in range(B):
        L = int(accept_len[r])
        keep = L + 1
        c0 = int(ctx[r])
        have = (c0 + P - 1) // P
        need = (c0 + keep + P - 1) // P
        for k in range(have, need):
            if top == 0 or k >= pt.shape[1]:
                raise NoSpace(f"request {r}: no free page or page-table row full")
            top -= 1
            pt[r, k] = int(free_pages[top])
        for i in range(keep):
            pos = c0 + i
            page = int(pt[r, pos // P])
            kc[page, pos % P] = k_new[int(cu_seqlens[r]) + i]
            if vc is not None:
                vc[page, pos % P] = v_new[int(cu_seqlens[r]) + i]
        ctx[r] = c0 + keep
        anc[r] = int(out_tok[r])
        committed[r, :L] = draft_tok[r, :L]
        committed[r, L] = int(out_tok[r])
        ncom[r] = keep
    return Compact(pt, ctx, anc, top, committed, ncom, kc, vc)


# ----------------------------------------------------------------------------
# 7. Calibration of the confidence head: labelled samples, ECE, STS refit
# ----------------------------------------------------------------------------

def calib_samples(survival, a_hat, windows, cap_len, mode, gamma):
    """Labelled accept outcomes of one step, per draft position ([csdn] §5
    "可观测性": per-request confidence and calibration metrics such as ECE;
    [notes] §07: the head's cumulative survival a_j predicts that the prefix
    1..j is accepted).

    Position j (1-based) of request r is verified iff j <= v_r (v_r = w_r in
    compact/static mode, gamma in cap-accept mode); its label is y = 1 iff the
    accepted prefix over the verified positions reaches it, j <= cap_r.
    Returns, per position j (0-based index), the list of (a_{r,j}, a_hat_{r,j}, y)
    in request order.
    """
    B = len(windows)
    out = [[] for _ in range(gamma)]
    for r in range(B):
        v = gamma if mode == CAP_ACCEPT else int(windows[r])
        for j in range(v):
            y = 1 if j + 1 <= int(cap_len[r]) else 0
            out[j].append((F32(survival[r, j]), F32(a_hat[r, j]), y))
    return out


def ece(samples, n_bins):
    """Expected calibration error of the calibrated survival a_hat against the
    labels, over all positions' samples: equal-width bins over [0, 1], bin of p
    = min(floor(p * n_bins), n_bins - 1), and
    ECE = sum_b (n_b / N) |mean(y in b) - mean(p in b)| = (1/N) sum_b |sum y - sum p|.
    fp64 sums.  Returns (ece, counts, sum_p, sum_y) per bin; ece = 0 when N = 0.
    """
    cnt = np.zeros(n_bins, dtype=np.int64)
    sp = np.zeros(n_bins, dtype=np.float64)
    sy = np.zeros(n_bins, dtype=np.float64)
    for pos in samples:
        for (_, p, y) in pos:
            b = min(int(math.floor(float(p) * n_bins)), n_bins - 1)
            cnt[b] += 1
            sp[b] += float(p)
            sy[b] += y
    N = int(cnt.sum())
    e = float(np.abs(sy - sp).sum() / N) if N else 0.0
    return e, cnt, sp, sy


STS_LOG_BETA_RANGE = (-math.log(64.0), math.log(64.0))


def sts_fit(samples_j, iters):
    """Refit one position's STS temperature from labelled samples ([notes] §07,
    Sequential Temperature Scaling: a_hat = sigmoid(logit(a) / T)).

    T minimises the binary cross-entropy of sigmoid(beta z) against the labels,
    beta = 1/T, z = logit(a) = log a - log1p(-a) (samples with a <= 0 or a >= 1
    have an infinite logit and are left out).  The loss is convex in beta, so its
    derivative g(beta) = sum (sigmoid(beta z) - y) z is increasing; the root is
    found by `iters` bisections of log beta over [log 1/64, log 64] (beta outside
    the range is clamped to it): g(mid) > 0 moves the upper end, else the lower.
    fp64 throughout.  No usable sample: T = 1.
    """
    zs, ys = [], []
    for (a, _, y) in samples_j:
        a = float(a)
        if 0.0 < a < 1.0:
            zs.append(math.log(a) - math.log1p(-a))
            ys.append(float(y))
    if not zs:
        return F32(1.0)
    z = np.array(zs, dtype=np.float64)
    y = np.array(ys, dtype=np.float64)
    lo, hi = STS_LOG_BETA_RANGE
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        beta = math.exp(mid)
        g = 0.0
        for zi, yi in zip(z, y):                     # plain loop: order is sample order
            t = beta * zi
            sig = 1.0 / (1.0 + math.exp(-t)) if t >= 0 else math.exp(t) / (1.0 + math.exp(t))
            g += (sig - yi) * zi
        if g > 0.0:
            hi = mid
        else:
            lo = mid
    return F32(1.0 / math.exp(0.5 * (lo + hi)))


# ----------------------------------------------------------------------------
# 8. The whole step
# ----------------------------------------------------------------------------

def step(inp: dict, mode: int, packed: dict | None = None, with_attention: bool = True,
         attention_requests=None) -> dict:
    """One verification step: schedule -> pack -> verify attention -> accept ->
    compact ([notes] §09 cycle; [lesson] "Confidence scheduler" through
    "Zero-overhead scheduling").  ``inp`` holds numpy arrays as drawn by the
    input generator; ``packed`` holds the packed per-row tensors (the caller
    lays the dense ones out with the oracle's own cu_seqlens).
    ``attention_requests`` restricts attention to a sample of requests.
    """
    wl = inp["workload"]
    sch = schedule(inp["conf"], inp["conf_is_logit"], inp["sts_temp"], inp["cost_table"],
                   wl.max_tokens, mode)
    pk = pack(sch.windows, inp["ctx_len"], inp["anchor"], inp["draft_tok"], inp["tiers"], mode,
              wl.gamma)
    out = {"schedule": sch, "pack": pk}
    if packed is None:
        return out
    if with_attention:
        out["attn"] = attention_for(inp, packed, pk.cu_seqlens, attention_requests)
    acc = accept(packed["p_target"], inp["p_draft"], inp["draft_tok"], inp["uniforms"],
                 inp["exp_noise"], sch.windows, pk.cu_seqlens, mode, wl.gamma)
    out["accept"] = acc
    out["compact"] = compact(packed["k_new"], packed.get("v_new"), pk.cu_seqlens, acc.accept_len,
                             acc.out_tok, inp["draft_tok"], wl.page_size, inp["page_table"],
                             inp["ctx_len"], inp["anchor"], inp["free_pages"],
                             int(np.asarray(inp["free_top"]).reshape(-1)[0]), inp["k_cache"],
                             inp["v_cache"])
    return out


def attention_for(inp, packed, cu_seqlens, requests=None):
    """Attention for all requests, or only ``requests`` (rows of the others are
    left as NaN)."""
    wl = inp["workload"]
    B = wl.B
    reqs = range(B) if requests is None else list(requests)
    M = int(cu_seqlens[B])
    o = np.full((M, wl.Hq, wl.d_v), np.nan)
    lse = np.full((M, wl.Hq), np.nan)
    for r in reqs:
        c0, c1 = int(cu_seqlens[r]), int(cu_seqlens[r + 1])
        sub_cu = np.array([0, c1 - c0], dtype=np.int64)
        if wl.attn == "gqa":
            o_r, l_r = verify_attention_gqa(
                packed["q"][c0:c1], packed["k_new"][c0:c1], packed["v_new"][c0:c1],
                inp["k_cache"], inp["v_cache"], inp["page_table"][r:r + 1],
                inp["ctx_len"][r:r + 1], sub_cu, wl.Hq, wl.Hkv, 1.0 / math.sqrt(wl.d_qk))
        else:
            o_r, l_r = verify_attention_mla(
                packed["q"][c0:c1], packed["k_new"][c0:c1], inp["k_cache"],
                inp["page_table"][r:r + 1], inp["ctx_len"][r:r + 1], sub_cu, wl.d_v,
                1.0 / math.sqrt(wl.d_qk))
        o[c0:c1], lse[c0:c1] = o_r, l_r
    return o, lse


# ----------------------------------------------------------------------------
# 9. Draft-side sampling with a Markov head
# ----------------------------------------------------------------------------

def markov_draft(U, W1, W2, anchor, exp_noise, tokens_given=None):
    """The drafter's block sampled position by position ([notes] §05 "Core
    Innovation A", 5.1-5.3): the parallel backbone gives base logits U_k for every
    position k of the block, the sequential Markov head adds a bias that depends only
    on the previous token, B(x_{k-1}, v) = (W1 W2)[x_{k-1}, v] (low rank, r = 256):

        p_k(v | x_{<k}) = exp(U_k(v) + B(x_{k-1}, v)) / sum_u exp(U_k(u) + B(x_{k-1}, u))

    with x_0 the anchor (the last committed token).  x_k is drawn by the Gumbel-max
    in its exponential-race form, argmax_v p_k(v) / e_k(v) with e ~ Exp(1) given
    (lowest index on ties; [notes] §02 sampling, reading A11).

    U fp32 [B, gamma, V]; W1 [V, r] and W2 [r, V] (bf16 values, given as float);
    anchor int [B]; exp_noise fp32 [B, gamma, V].  fp64 throughout (the bias is the
    plain product of the previous token's W1 row with W2).  ``tokens_given``
    (int [B, gamma], optional) makes position k condition on tokens_given[:, k-1]
    instead of the oracle's own draw, so a chain can follow another sampler's tokens.
    Returns (tokens int32 [B, gamma], p fp64 [B, gamma, V], keys fp64 [B, gamma, V]).
    """
    U = np.asarray(U, dtype=np.float64)
    W1 = np.asarray(W1, dtype=np.float64)
    W2 = np.asarray(W2, dtype=np.float64)
    e = np.asarray(exp_noise, dtype=np.float64)
    B, gamma, V = U.shape
    tokens = np.zeros((B, gamma), dtype=np.int32)
    P = np.zeros((B, gamma, V), dtype=np.float64)
    K = np.zeros((B, gamma, V), dtype=np.float64)
    for r in range(B):
        prev = int(anchor[r])
        for k in range(gamma):
            logits = U[r, k] + W1[prev] @ W2
            z = logits - logits.max()
            w = np.exp(z)
            p = w / w.sum()
            keys = np.where(p > 0.0, p / e[r, k], -np.inf)
            x = int(np.argmax(keys))          # first maximum: lowest index on ties
            P[r, k], K[r, k] = p, keys
            tokens[r, k] = x
            prev = x if tokens_given is None else int(tokens_given[r, k])
    return tokens, P, K



# ----------------------------------------------------------------------------
# 10. Block-accept estimator: the uncut cap from inside a compact run
# ----------------------------------------------------------------------------

def block_accept_estimate(p_target, p_draft, draft_tok, uniforms, windows, cu_seqlens,
                          accept_len, cap_len, mode, gamma):
    """The accepted-prefix length a full-block verification would have seen (the
    cap that cap-accept exposes), recovered inside the step ([csdn] 5 "可观测性":
    compact verifies only the window, so the uncut cap is censored; the estimator
    recovers an interval for it from tensors the run already has).

    Reading A29.  Compact mode, request r with window w and L accepted drafts:
      * L < w: a draft inside the window was rejected, the cap is L;
      * L = w = gamma: the whole block was verified and accepted, the cap is gamma;
      * L = w < gamma: the step holds the target row of position w + 1 (the bonus
        row, packed row cu_seqlens[r] + w) and the drafter's row of that position,
        so the test a full-block run makes at w + 1 is made here with the same
        operands (u_{w+1} p_d(d_{w+1}) <= p_t(d_{w+1}), fp32):
          rejected -> the cap is w;  accepted -> the cap lies in [w + 1, gamma].
    Static and cap-accept modes verify the whole block: the cap is cap_len.

    Returns (cap_lo, cap_hi) int32 [B]; cap_lo == cap_hi where the cap is known.
    """
    B = len(windows)
    lo = np.zeros(B, dtype=np.int32)
    hi = np.zeros(B, dtype=np.int32)
    for r in range(B):
        if mode != COMPACT:
            lo[r] = hi[r] = int(cap_len[r])
            continue
        w, L = int(windows[r]), int(accept_len[r])
        if L < w or w == gamma:
            lo[r] = hi[r] = L
            continue
        x = int(draft_tok[r, w])                       # d_{w+1}
        pt = F32(p_target[int(cu_seqlens[r]) + w, x])  # target row of position w + 1
        pd = F32(p_draft[r, w, x])
        if F32(F32(uniforms[r, w]) * pd) <= pt:
            lo[r], hi[r] = w + 1, gamma
        else:
            lo[r] = hi[r] = w
    return lo, hi

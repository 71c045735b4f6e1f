"""Seeded synthetic inputs for the DSpark verification step.

This module holds only workload definitions and random-number draws.  It holds
none of the method's arithmetic (no survival product, no scheduling, no
attention, no acceptance, no compaction); both the CUDA path and the oracle
consume what it returns.

Every tensor is drawn from its own torch.Generator, seeded from (seed, name), on
the device it is asked for.  Small workloads are drawn on the CPU and copied, so
CPU-only tests and GPU tests see identical values for them.

Shapes follow the five workloads of the DSpark verification study:

* ``tiny``      B=4,   gamma=6,  GQA 8/2 heads x 128, ctx U[64,256],   V=1024
* ``qwen3_8b``  B=32,  gamma=8,  GQA 32/8 heads x 128, ctx U[1024,4096], V=151936 (fp32 p)
* ``mixed256``  B=256, gamma=16, GQA 40/8 heads x 128, ctx lognormal(2048,0.6)
                clipped [512,8192], three confidence classes, V=151936 (bf16 p)
* ``mla``       B=64,  gamma=8,  128 heads sharing one 576-d latent (v 512),
                ctx U[4096,32768], page 64, V=129280
* ``sweep``     Qwen3-8B shape, gamma=16, B in {1,8,32,128,256}, ctx 2048,
                confidence mean in {.95,.85,.70}, cost slope in {.05,.19,.5}
"""
from __future__ import annotations

import dataclasses
import math
import zlib
from typing import Optional

import torch

MODE_COMPACT, MODE_STATIC, MODE_CAP_ACCEPT = 0, 1, 2
MODE_NAMES = {"compact": MODE_COMPACT, "static": MODE_STATIC, "cap_accept": MODE_CAP_ACCEPT}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    gamma: int
    attn: str                      # "gqa" or "mla"
    Hq: int
    Hkv: int                       # 1 for mla (one shared latent)
    d_qk: int
    d_v: int
    page_size: int
    ctx: tuple                     # ("uniform", lo, hi) | ("lognormal", median, sigma, lo, hi) | ("const", n)
    conf: tuple                    # ("logit", mean, std) | ("classes", (means...), std)
    vocab: int
    p_dtype: str                   # "f32" or "bf16"
    target_logit_std: float
    draft_noise_std: float
    tiers: tuple
    sts_lo: float = 1.0
    sts_hi: float = 1.5
    cost_bias_ms: float = 20.0
    cost_theta_ms: float = 0.19
    modes: tuple = ("compact",)

    @property
    def group(self) -> int:
        return self.Hq // self.Hkv

    @property
    def max_tokens(self) -> int:
        return max(self.tiers)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def pow2_tiers(lo: int, upto: int) -> tuple:
    t, out = lo, []
    while True:
        out.append(t)
        if t >= upto:
            return tuple(out)
        t *= 2


WORKLOADS = {
    "tiny": Workload(
        name="tiny", B=4, gamma=6, attn="gqa", Hq=8, Hkv=2, d_qk=128, d_v=128, page_size=16,
        ctx=("uniform", 64, 256), conf=("logit", 1.0, 1.0), vocab=1024, p_dtype="f32",
        target_logit_std=2.0, draft_noise_std=0.5, tiers=pow2_tiers(8, 4 * 7)),
    "qwen3_8b": Workload(
        name="qwen3_8b", B=32, gamma=8, attn="gqa", Hq=32, Hkv=8, d_qk=128, d_v=128, page_size=16,
        ctx=("uniform", 1024, 4096), conf=("logit", 1.5, 1.0), vocab=151936, p_dtype="f32",
        target_logit_std=3.0, draft_noise_std=0.7, tiers=pow2_tiers(8, 512)),
    "mixed256": Workload(
        name="mixed256", B=256, gamma=16, attn="gqa", Hq=40, Hkv=8, d_qk=128, d_v=128, page_size=16,
        ctx=("lognormal", 2048.0, 0.6, 512, 8192), conf=("classes", (0.93, 0.85, 0.75), 0.05),
        vocab=151936, p_dtype="bf16", target_logit_std=3.0, draft_noise_std=0.7,
        tiers=pow2_tiers(8, 256 * 17), modes=("compact", "static", "cap_accept")),
    "mla": Workload(
        name="mla", B=64, gamma=8, attn="mla", Hq=128, Hkv=1, d_qk=576, d_v=512, page_size=64,
        ctx=("uniform", 4096, 32768), conf=("logit", 1.2, 1.0), vocab=129280, p_dtype="f32",
        target_logit_std=3.0, draft_noise_std=0.7, tiers=pow2_tiers(8, 64 * 9)),
    "sweep": Workload(
        name="sweep", B=32, gamma=16, attn="gqa", Hq=32, Hkv=8, d_qk=128, d_v=128, page_size=16,
        ctx=("const", 2048), conf=("classes", (0.85,), 0.05), vocab=151936, p_dtype="f32",
        target_logit_std=3.0, draft_noise_std=0.7, tiers=pow2_tiers(4, 4096),
        modes=("compact", "static", "cap_accept")),
}

SWEEP_B = (1, 8, 32, 128, 256)
SWEEP_CONF_MEANS = (0.95, 0.85, 0.70)
SWEEP_THETA = (0.05, 0.19, 0.5)


def sweep_point(B: int, conf_mean: float, theta: float) -> Workload:
    return WORKLOADS["sweep"].replace(
        name=f"sweep_B{B}_c{conf_mean}_t{theta}", B=B, conf=("classes", (conf_mean,), 0.05),
        cost_theta_ms=theta)


def _gen(seed: int, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + zlib.crc32(name.encode())) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def _uniform_open01_f32(shape, g, device) -> torch.Tensor:
    """U = (2k + 1) 2^-24 with k uniform on [0, 2^23): the 2^23 odd multiples of 2^-24.

    An odd integer below 2^24 has at most 24 significant bits, so every value is an
    exact fp32 number, the smallest 2^-24 and the largest 1 - 2^-24: never 0, never 1
    (so -log U is finite and strictly positive).
    """
    k = torch.randint(0, 1 << 23, shape, generator=g, device=device, dtype=torch.int64)
    return ((2 * k + 1).to(torch.float64) * 2.0 ** -24).to(torch.float32)


def _ctx_lengths(wl: Workload, g, device) -> torch.Tensor:
    kind = wl.ctx[0]
    if kind == "uniform":
        lo, hi = wl.ctx[1], wl.ctx[2]
        return torch.randint(lo, hi + 1, (wl.B,), generator=g, device=device, dtype=torch.int64)
    if kind == "lognormal":
        med, sig, lo, hi = wl.ctx[1:]
        z = torch.randn((wl.B,), generator=g, device=device, dtype=torch.float64)
        return torch.clamp(torch.round(med * torch.exp(sig * z)), lo, hi).to(torch.int64)
    if kind == "const":
        return torch.full((wl.B,), wl.ctx[1], device=device, dtype=torch.int64)
    raise ValueError(kind)


def _confidence(wl: Workload, g, device):
    kind = wl.conf[0]
    if kind == "logit":
        z = wl.conf[1] + wl.conf[2] * torch.randn((wl.B, wl.gamma), generator=g, device=device,
                                                  dtype=torch.float64)
        return z.to(torch.float32), 1
    if kind == "classes":
        means, std = wl.conf[1], wl.conf[2]
        cls = torch.arange(wl.B, device=device) % len(means)
        mu = torch.tensor(means, device=device, dtype=torch.float64)[cls][:, None]
        c = mu + std * torch.randn((wl.B, wl.gamma), generator=g, device=device, dtype=torch.float64)
        c = torch.clamp(c, 1e-6, 1.0 - 1e-6)
        return c.to(torch.float32), 0
    raise ValueError(kind)


def gen_device(wl: Workload) -> str:
    """Where the draws for this workload are made when a GPU is in use."""
    small = wl.B * (wl.gamma + 1) * wl.vocab <= (1 << 22)
    return "cpu" if small else "cuda"


@torch.no_grad()
def make_inputs(wl: Workload, seed: int = 0, device: str = "cpu",
                extra_free_pages: Optional[int] = None, ctx_override=None) -> dict:
    """Draw one verification step's inputs for workload ``wl``.

    Per-position tensors are dense over the block: row (r, i) of a ``*_dense``
    tensor is what the target model would hand the verify step for request r,
    in-block position i (i = 0 is the anchor, i >= 1 the draft token d_i).  The
    caller lays them out head-to-tail with ``to_packed`` once cu_seqlens is
    known.
    """
    dev = device
    B, gam, P = wl.B, wl.gamma, wl.page_size
    out = {"workload": wl, "seed": seed}

    conf, is_logit = _confidence(wl, _gen(seed, "conf", dev), dev)
    out["conf"], out["conf_is_logit"] = conf, is_logit
    out["sts_temp"] = torch.linspace(wl.sts_lo, wl.sts_hi, gam, dtype=torch.float64,
                                     device=dev).to(torch.float32)
    cost_len = max(wl.max_tokens, B * (gam + 1)) + 2
    m = torch.arange(cost_len, dtype=torch.float64, device=dev)
    out["cost_table"] = (wl.cost_bias_ms + wl.cost_theta_ms * m).to(torch.float32)
    out["tiers"] = torch.tensor(wl.tiers, dtype=torch.int32)

    ctx = _ctx_lengths(wl, _gen(seed, "ctx", dev), dev)
    if ctx_override is not None:
        ctx = torch.as_tensor(list(ctx_override), dtype=torch.int64, device=dev)
    out["ctx_len"] = ctx.to(torch.int32)
    # Paged cache: every request's committed context lives in pages drawn at random
    # from one pool; the rest of the pool is the free-page stack.
    pages_per_req = (ctx + P - 1) // P
    max_ctx_after = int(ctx.max().item()) + gam + 1
    max_pages = (max_ctx_after + P - 1) // P + 1
    n_used = int(pages_per_req.sum().item())
    grow = B * ((gam + 1 + P - 1) // P + 1)
    n_free = grow if extra_free_pages is None else extra_free_pages
    n_pages = n_used + n_free
    perm = torch.randperm(n_pages, generator=_gen(seed, "pages", dev), device=dev).to(torch.int32)
    page_table = torch.full((B, max_pages), -1, dtype=torch.int32, device=dev)
    starts = torch.cumsum(pages_per_req, 0) - pages_per_req
    col = torch.arange(max_pages, device=dev)[None, :]
    used = col < pages_per_req[:, None]
    idx = (starts[:, None] + col).clamp(max=n_pages - 1)
    page_table = torch.where(used, perm[idx.long()], page_table)
    out["page_table"] = page_table.contiguous()
    # never an empty tensor: an exhausted stack is free_top = 0 over a 1-entry buffer
    out["free_pages"] = (perm[n_used:].contiguous() if n_free > 0
                         else torch.zeros(1, dtype=torch.int32, device=dev))
    out["free_top"] = torch.tensor([n_free], dtype=torch.int32, device=dev)
    out["n_pages"] = n_pages

    gk = _gen(seed, "kv", dev)
    if wl.attn == "gqa":
        out["k_cache"] = torch.randn((n_pages, P, wl.Hkv, wl.d_qk), generator=gk, device=dev,
                                     dtype=torch.float32).to(torch.bfloat16)
        out["v_cache"] = torch.randn((n_pages, P, wl.Hkv, wl.d_v), generator=gk, device=dev,
                                     dtype=torch.float32).to(torch.bfloat16)
        out["k_new_dense"] = torch.randn((B, gam + 1, wl.Hkv, wl.d_qk), generator=gk, device=dev,
                                         dtype=torch.float32).to(torch.bfloat16)
        out["v_new_dense"] = torch.randn((B, gam + 1, wl.Hkv, wl.d_v), generator=gk, device=dev,
                                         dtype=torch.float32).to(torch.bfloat16)
    else:
        out["k_cache"] = torch.randn((n_pages, P, wl.d_qk), generator=gk, device=dev,
                                     dtype=torch.float32).to(torch.bfloat16)
        out["v_cache"] = None
        out["k_new_dense"] = torch.randn((B, gam + 1, wl.d_qk), generator=gk, device=dev,
                                         dtype=torch.float32).to(torch.bfloat16)
        out["v_new_dense"] = None
    out["q_dense"] = torch.randn((B, gam + 1, wl.Hq, wl.d_qk), generator=_gen(seed, "q", dev),
                                 device=dev, dtype=torch.float32).to(torch.bfloat16)

    # Target / draft distributions: softmax of Gaussian logits; the draft's logits are
    # the target's plus independent Gaussian noise.  Drawn request by request to bound
    # the temporary memory.
    pdt = torch.float32 if wl.p_dtype == "f32" else torch.bfloat16
    V = wl.vocab
    p_t = torch.empty((B, gam + 1, V), dtype=pdt, device=dev)
    p_d = torch.empty((B, gam, V), dtype=pdt, device=dev)
    draft = torch.empty((B, gam), dtype=torch.int32, device=dev)
    gt, gd, gs = _gen(seed, "p_target", dev), _gen(seed, "p_draft", dev), _gen(seed, "drafts", dev)
    chunk = max(1, (1 << 24) // ((gam + 1) * V))
    for r0 in range(0, B, chunk):
        r1 = min(B, r0 + chunk)
        lt = wl.target_logit_std * torch.randn((r1 - r0, gam + 1, V), generator=gt, device=dev,
                                               dtype=torch.float32)
        ld = lt[:, :gam, :] + wl.draft_noise_std * torch.randn((r1 - r0, gam, V), generator=gd,
                                                             device=dev, dtype=torch.float32)
        pt = torch.softmax(lt, dim=-1)
        pd = torch.softmax(ld, dim=-1)
        p_t[r0:r1] = pt.to(pdt)
        p_d[r0:r1] = pd.to(pdt)
        # draft token i (1-based) is drawn from the draft distribution at position i
        flat = pd.to(pdt).to(torch.float32).reshape(-1, V)
        draft[r0:r1] = torch.multinomial(flat, 1, generator=gs).reshape(r1 - r0, gam).to(torch.int32)
        del lt, ld, pt, pd, flat
    # p_dense row (r, i) is the target's distribution for in-block position i+1,
    # i.e. the output of verify row i.
    out["p_target_dense"] = p_t
    out["p_draft"] = p_d
    out["draft_tok"] = draft
    out["anchor"] = torch.randint(0, V, (B,), generator=_gen(seed, "anchor", dev), device=dev,
                                  dtype=torch.int32)
    out["uniforms"] = _uniform_open01_f32((B, gam), _gen(seed, "uniforms", dev), dev)
    u2 = _uniform_open01_f32((B, V), _gen(seed, "exp_noise", dev), dev)
    out["exp_noise"] = (-torch.log(u2.to(torch.float64))).to(torch.float32)
    return out


# Markov-head draft sampling: the drafter's block of base logits and a random head.
MARKOV_WORKLOADS = {
    # Qwen3-8B vocabulary, the verification workload's batch and block
    "markov_qwen3_8b": dict(B=32, gamma=8, V=151936),
    # parity cases: one request; a ragged column group; one tile per CTA; a partly
    # filled last round of tiles over two launches; sixteen tiles per CTA
    "markov_one": dict(B=1, gamma=1, V=1024),
    "markov_small": dict(B=5, gamma=6, V=1024),
    "markov_g32": dict(B=32, gamma=6, V=4096),
    "markov_ragged": dict(B=37, gamma=4, V=40960),
    "markov_wide": dict(B=20, gamma=2, V=311296),
}


@torch.no_grad()
def make_markov_inputs(B: int, gamma: int, V: int, seed: int = 0, device: str = "cpu",
                       rank: int = 256, u_std: float = 3.0, w_std: float = 0.25) -> dict:
    """Base logits U ~ N(0, u_std^2) fp32 [B, gamma, V]; head weights W1 [V, rank] and
    W2 [rank, V] ~ N(0, w_std^2) rounded to bf16 (with rank 256 and w_std 0.25 the bias
    of a token has standard deviation about 1); anchors uniform on [0, V); exp_noise
    = -ln(U) with U uniform on the open interval (Exp(1) draws), fp32 [B, gamma, V]."""
    dev = torch.device(device)
    out = {}
    out["U"] = u_std * torch.randn((B, gamma, V), generator=_gen(seed, "markov_U", dev), device=dev,
                                   dtype=torch.float32)
    out["W1"] = (w_std * torch.randn((V, rank), generator=_gen(seed, "markov_W1", dev), device=dev,
                                     dtype=torch.float32)).to(torch.bfloat16)
    out["W2"] = (w_std * torch.randn((rank, V), generator=_gen(seed, "markov_W2", dev), device=dev,
                                     dtype=torch.float32)).to(torch.bfloat16)
    out["anchor"] = torch.randint(0, V, (B,), generator=_gen(seed, "markov_anchor", dev), device=dev,
                                  dtype=torch.int32)
    u = _uniform_open01_f32((B, gamma, V), _gen(seed, "markov_noise", dev), dev)
    out["exp_noise"] = (-torch.log(u.to(torch.float64))).to(torch.float32)
    return out


def to_packed(dense: torch.Tensor, cu_seqlens: torch.Tensor, total_rows: int) -> torch.Tensor:
    """Lay per-position rows out head-to-tail: row cu_seqlens[r] + i <- dense[r, i].

    Rows past cu_seqlens[B] (tier padding) are zero.  Pure indexing.
    """
    cu = cu_seqlens.to(torch.int64).to(dense.device)
    B = dense.shape[0]
    n = cu[1:] - cu[:-1]
    out = torch.zeros((total_rows,) + tuple(dense.shape[2:]), dtype=dense.dtype, device=dense.device)
    r = torch.repeat_interleave(torch.arange(B, device=dense.device), n)
    i = torch.arange(int(cu[-1].item()), device=dense.device) - cu[:-1][r]
    out[: int(cu[-1].item())] = dense[r, i]
    return out


def cap_rows(wl: Workload) -> int:
    """Upper bound on verify rows a step can occupy (largest tier, or B*(gamma+1))."""
    return max(wl.max_tokens, wl.B * (wl.gamma + 1))

"""Glue between the seeded inputs and the CUDA library: device placement, packed
per-row layouts and one full verification step through the C ABI.

Used by the GPU tests, ``__graft_entry__.smoke`` and ``bench.py``.  It holds no
arithmetic of the method: every step runs in libdspark.so.
"""
from __future__ import annotations

import math

import torch

import speculative_decoding_verification_dspark_gb300 as dspark
import workloads as W

STATE_KEYS = ("page_table", "ctx_len", "anchor", "free_top", "k_cache", "v_cache")


def device_inputs(inp: dict, device="cuda") -> dict:
    """Everything the step reads, on the device (packed buffers are added later)."""
    wl = inp["workload"]
    d = {}
    for k, v in inp.items():
        if isinstance(v, torch.Tensor):
            # state is updated in place by compact: never alias the caller's tensors
            d[k] = v.to(device, copy=k in STATE_KEYS).contiguous()
        else:
            d[k] = v
    d["max_tokens"] = wl.max_tokens
    d["scale"] = 1.0 / math.sqrt(wl.d_qk)
    return d


def make_step(wl: W.Workload, max_splits: int = 8) -> dspark.VerifyStep:
    pdt = torch.float32 if wl.p_dtype == "f32" else torch.bfloat16
    return dspark.VerifyStep(wl.B, wl.gamma, wl.Hq, wl.Hkv, wl.d_qk, wl.d_v, wl.vocab,
                             W.cap_rows(wl), pdt, max_splits=max_splits)


def attach_packed(d: dict, cu_seqlens_cpu: torch.Tensor, max_rows: int) -> None:
    """Lay the per-position tensors out as the packed rows the target would hand over."""
    d["q"] = W.to_packed(d["q_dense"], cu_seqlens_cpu, max_rows)
    d["k_new"] = W.to_packed(d["k_new_dense"], cu_seqlens_cpu, max_rows)
    if d.get("v_new_dense") is not None:
        d["v_new"] = W.to_packed(d["v_new_dense"], cu_seqlens_cpu, max_rows)
    else:
        d["v_new"] = None
    d["p_target"] = W.to_packed(d["p_target_dense"], cu_seqlens_cpu, max_rows)


def snapshot_state(d: dict) -> dict:
    return {k: (d[k].clone() if isinstance(d.get(k), torch.Tensor) else d.get(k)) for k in STATE_KEYS}


def restore_state(d: dict, snap: dict) -> None:
    for k, v in snap.items():
        if isinstance(v, torch.Tensor):
            d[k].copy_(v, non_blocking=True)


def prepare(inp: dict, mode: int, step: dspark.VerifyStep | None = None, device="cuda"):
    """Device inputs + a schedule/pack pass to learn the packed layout; returns (d, step)."""
    wl = inp["workload"]
    d = device_inputs(inp, device)
    if step is None:
        step = make_step(wl)
    step.schedule(d, mode)
    step.pack(d, mode)
    torch.cuda.synchronize()
    attach_packed(d, step.cu_seqlens.cpu(), step.max_rows)
    return d, step


def run_step(inp: dict, mode: int, device="cuda") -> dict:
    """One full step through the C ABI; returns host copies of every output."""
    d, step = prepare(inp, mode, device=device)
    step.run(d, mode)
    err = dspark.read_device_error()
    torch.cuda.synchronize()
    out = {
        "device_error": err,
        "windows": step.windows.cpu(), "a_hat": step.a_hat.cpu(), "M": int(step.M.item()),
        "E": float(step.E.item()), "cu_seqlens": step.cu_seqlens.cpu(),
        "M_pack": int(step.M_pack.item()), "tier": int(step.tier.item()),
        "row_req": step.row_req.cpu(), "row_pos": step.row_pos.cpu(), "row_tok": step.row_tok.cpu(),
        "out": step.out.cpu(), "lse": step.lse.cpu(),
        "accept_len": step.accept_len.cpu(), "cap_len": step.cap_len.cpu(),
        "out_tok": step.out_tok.cpu(), "fallback": step.fallback.cpu(), "cstar": step.cstar.cpu(),
        "committed": step.committed.cpu(), "n_committed": step.n_committed.cpu(),
        "page_table": d["page_table"].cpu(), "ctx_len": d["ctx_len"].cpu(),
        "anchor": d["anchor"].cpu(), "free_top": int(d["free_top"].item()),
        "k_cache": d["k_cache"], "v_cache": d.get("v_cache"),
    }
    return out

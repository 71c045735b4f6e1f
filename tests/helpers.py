"""Test plumbing: torch inputs -> numpy for the oracle; packed per-row layouts."""
import numpy as np
import torch

import workloads as W


def to_np(x):
    if isinstance(x, torch.Tensor):
        t = x.detach().cpu()
        if t.dtype == torch.bfloat16:
            t = t.to(torch.float32)
        return t.numpy()
    return x


def np_inputs(inp: dict) -> dict:
    return {k: to_np(v) for k, v in inp.items()}


def packed_inputs(inp: dict, cu_seqlens, total_rows: int) -> dict:
    """Per-row tensors laid out head-to-tail with the given cu_seqlens (torch)."""
    cu = torch.as_tensor(np.asarray(cu_seqlens), dtype=torch.int32)
    out = {
        "q": W.to_packed(inp["q_dense"], cu, total_rows),
        "k_new": W.to_packed(inp["k_new_dense"], cu, total_rows),
        "p_target": W.to_packed(inp["p_target_dense"], cu, total_rows),
    }
    if inp.get("v_new_dense") is not None:
        out["v_new"] = W.to_packed(inp["v_new_dense"], cu, total_rows)
    return out


def oracle_step(inp: dict, mode: int, with_attention=True, attention_requests=None):
    from oracle import dspark_oracle as O
    npi = np_inputs(inp)
    base = O.step(npi, mode)
    pk = base["pack"]
    packed = {k: to_np(v) for k, v in packed_inputs(inp, pk.cu_seqlens, pk.tier).items()}
    return O.step(npi, mode, packed, with_attention=with_attention,
                  attention_requests=attention_requests), packed

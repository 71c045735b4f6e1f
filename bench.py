"""Benchmark of the DSpark confidence-scheduled ragged verification step on GB300.

Default: the Qwen3-8B-shaped workload (B=32, gamma=8, 32/8 heads x 128, context
U[1024,4096], page 16, vocab 151936 fp32 probabilities, compact mode) on one GPU.
One step = schedule -> pack -> verify attention -> accept -> compact over one
batch, captured once in a CUDA graph and replayed; the small mutable state
(page table, ctx_len, anchor, free-stack top) is restored inside the step so
that every step does identical work.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload qwen3_8b|mixed256|mla|tiny] [--mode compact|static|cap_accept]

Prints one JSON line (rank 0).
"""
from __future__ import annotations

import os

# The CPU oracle (baseline leg and reference arm) runs single-threaded.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import hashlib
import json
import math
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "verify steps/s & packed tokens/s at B=1..256, % of HBM roofline per kernel"
UNIT = "verify steps/s"
KERNELS_PER_STEP = 10   # schedule 2, pack + work list 1, attention 2, accept 3, compact 2
PROFILES = os.path.join(ROOT, "profiles")
_CSRC = os.path.join(ROOT, "speculative_decoding_verification_dspark_gb300", "csrc")
# sources whose change invalidates a committed DRAM-traffic figure
_ATTN_COMMON = ("verify_attn.cu", "worklist.cuh", "attn.h", "ptx.cuh", "common.cuh")


def attn_src(wl):
    """The attention call's sources for this workload's head shape."""
    main = "verify_attn_mla.cu" if wl.attn == "mla" else "verify_attn_gqa.cu"
    return [os.path.join(_CSRC, f) for f in _ATTN_COMMON + (main,)]


ACCEPT_SRC = [os.path.join(_CSRC, f) for f in ("accept.cu", "common.cuh")]


def workload_desc(wl: W.Workload, mode: str) -> str:
    head = (f"GQA {wl.Hq}/{wl.Hkv} heads x {wl.d_qk}" if wl.attn == "gqa"
            else f"MLA {wl.Hq} heads, latent {wl.d_qk} (v {wl.d_v})")
    return (f"{wl.name}: B={wl.B} gamma={wl.gamma} {head} ctx={wl.ctx} page={wl.page_size} "
            f"V={wl.vocab} p={wl.p_dtype} mode={mode} tiers {wl.tiers[0]}..{wl.tiers[-1]}")


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)
        return dist
    return None


def max_over_ranks(x: float, dist, device) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, device):
    if dist is not None:
        dist.barrier()
    if device.type == "cuda":
        torch.cuda.synchronize()


# ------------------------------------------------------------------ clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ algorithmic bytes

def attn_bytes(wl, ctx, n_rows):
    """Bytes the verify attention must move: each request's K/V (cached + block rows)
    once, Q read (bf16), O (fp32) and lse (fp32) written."""
    ctx = np.asarray(ctx, np.int64)
    n = np.asarray(n_rows, np.int64)
    M = int(n.sum())
    if wl.attn == "gqa":
        kv = int(((ctx + n) * wl.Hkv * (wl.d_qk + wl.d_v) * 2).sum())
    else:
        kv = int(((ctx + n) * wl.d_qk * 2).sum())
    return kv + M * wl.Hq * (wl.d_qk * 2 + wl.d_v * 4 + 4)


def attn_flops(wl, ctx, n_rows):
    ctx = np.asarray(ctx, np.int64)
    n = np.asarray(n_rows, np.int64)
    # causal inside the block: row i sees ctx + i + 1 keys
    keys = (n * ctx + n * (n + 1) // 2)
    return int((2 * keys * wl.Hq * (wl.d_qk + wl.d_v)).sum())


def accept_bytes(wl, windows, n_rows, accept_len, mode):
    """Bytes the acceptance must move: for every position with a target row up to
    gamma, one p_t row and one p_d row (c*); the sampled row's noise row; a bonus
    row beyond gamma when the whole block was accepted."""
    s = 4 if wl.p_dtype == "f32" else 2
    V = wl.vocab
    tot = 0
    for r in range(wl.B):
        c_rows = min(int(n_rows[r]), wl.gamma)
        tot += 2 * c_rows * V * s + V * 4
        if int(accept_len[r]) == wl.gamma and int(windows[r]) == wl.gamma:
            tot += V * s
    return tot


# ------------------------------------------------------------------ GPU arm

def restore_pairs(d, keys):
    """(destination, saved copy) pairs that put the step's small mutable state back.
    When the tensors share a dtype they are moved into one buffer first (each a view
    at a 256-byte boundary), so the restore is a single copy."""
    ts = [d[k] for k in keys]
    if len({t.dtype for t in ts}) != 1 or len({t.device for t in ts}) != 1:
        return [(d[k], d[k].clone()) for k in keys]
    per = 256 // ts[0].element_size()
    offs, total = [], 0
    for t in ts:
        offs.append(total)
        total += (t.numel() + per - 1) // per * per
    flat = torch.zeros(total, dtype=ts[0].dtype, device=ts[0].device)
    for k, t, o in zip(keys, ts, offs):
        view = flat[o:o + t.numel()].view(t.shape)
        view.copy_(t)
        d[k] = view
    return [(flat, flat.clone())]


def gpu_arm(args, wl, mode, dist, world, rank, device, with_e2e=True):
    import harness
    import speculative_decoding_verification_dspark_gb300 as dspark

    inp = W.make_inputs(wl, seed=args.seed + rank, device=W.gen_device(wl))
    d, step = harness.prepare(inp, mode)
    snap = harness.snapshot_state(d)
    small = restore_pairs(d, ("page_table", "ctx_len", "anchor", "free_top"))
    stream = torch.cuda.Stream()
    # inputs, packed rows and the state snapshot were made on the default stream
    stream.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()

    def one_step():
        for dst, src in small:
            dst.copy_(src, non_blocking=True)
        step.run(d, mode)

    # eager warm-up (also compiles nothing: all kernels are precompiled)
    with torch.cuda.stream(stream):
        for _ in range(2):
            one_step()
    torch.cuda.synchronize()
    err = dspark.read_device_error()
    if err:
        raise RuntimeError(f"device error word {err:#x} during warm-up")

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        one_step()
    torch.cuda.synchronize()

    windows = step.windows.cpu().numpy()
    cu = step.cu_seqlens.cpu().numpy()
    n_rows = np.diff(cu)
    ctx0 = snap["ctx_len"].cpu().numpy()
    M = int(cu[-1])
    tier = int(step.tier.item())

    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist, device)
    with ClockSampler(device.index or 0) as clk:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            ev1.record(stream)
        ev1.synchronize()
    barrier(dist, device)
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(ms, dist, device)
    err = dspark.read_device_error()
    if err:
        raise RuntimeError(f"device error word {err:#x} in the timed region")
    acc_len = step.accept_len.cpu().numpy()

    # ---- per-kernel timing of the HBM-bound calls (graphs of repeated launches)
    def time_call(fn, reps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                fn()
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(args.kernel_iters):
                g.replay()
            b.record(stream)
        b.synchronize()
        return a.elapsed_time(b) * 1e3 / (reps * args.kernel_iters)  # us per call

    # the attention call of the step: over the work list its pack call built, from the
    # step's own state (restored, then packed once more)
    for dst, src in small:
        dst.copy_(src, non_blocking=True)
    step.pack_plan(d, mode)
    attn_us = time_call(lambda: step.attention_planned(d), 10)
    accept_us = time_call(lambda: step.accept(d, mode), 10)
    a_bytes = attn_bytes(wl, ctx0, n_rows)
    a_flops = attn_flops(wl, ctx0, n_rows)
    c_bytes = accept_bytes(wl, windows, n_rows, acc_len, mode)
    peaks = load_peaks()
    hbm = peaks.get("hbm_gbs")
    peak_src = "measured" if hbm else "fallback"
    hbm = hbm or 6800.0
    attn_gbs = a_bytes / (attn_us * 1e-6) / 1e9
    acc_gbs = c_bytes / (accept_us * 1e-6) / 1e9
    attn_tfs = a_flops / (attn_us * 1e-6) / 1e12
    traffic = load_traffic("verify_attn", wl.name, attn_src(wl))
    # the attention call is tensor-bound when its flops per algorithmic byte exceed the
    # ridge point of the measured peaks (the latent-KV shape), else HBM-bound
    tf_peak = peaks.get("bf16_tflops")
    tf_src = "measured" if tf_peak else "fallback"
    tf_peak = tf_peak or 1900.0
    tensor_bound = a_flops / max(a_bytes, 1) > tf_peak * 1e12 / (hbm * 1e9)
    if tensor_bound:
        roof = {"bound": "tensor", "kernel": "dspark_verify_attn (work list + main + combine)",
                "achieved": attn_tfs, "peak": tf_peak, "unit": "TFLOP/s", "frac": attn_tfs / tf_peak,
                "traffic": traffic, "algorithmic_flops": a_flops, "algorithmic_bytes": a_bytes,
                "us_per_launch": attn_us,
                "peak_source": f"{tf_src} bf16_tflops (burst cuBLAS GEMM; the kernel is timed alone)"}
    else:
        roof = {"bound": "hbm", "kernel": "dspark_verify_attn (work list + main + combine)",
                "achieved": attn_gbs, "peak": hbm, "unit": "GB/s", "frac": attn_gbs / hbm,
                "traffic": traffic, "algorithmic_bytes": a_bytes, "us_per_launch": attn_us,
                "peak_source": f"{peak_src} hbm_gbs (burst copy)"}

    err = dspark.read_device_error()
    if err:
        raise RuntimeError(f"device error word {err:#x} while timing the calls")
    # ---- end to end through the public API with host buffers
    e2e = e2e_arm(args, wl, mode, d, step, small, stream) if with_e2e else None
    err = dspark.read_device_error()
    if err:
        raise RuntimeError(f"device error word {err:#x} in the end-to-end arm")

    steps_per_s = args.steps / (ms_max / 1e3)
    value = world * args.steps / (ms_max / 1e3)
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "dtype_detail": "attention bf16 operands / fp32 accumulate and softmax; acceptance fp32",
        "data": "synthetic",
        "config": {"workload": workload_desc(wl, args.mode), "mode": args.mode,
                   "global_batch": wl.B * world, "packed_rows_M": M, "tier": tier,
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (no flush): KV %.2f GB, probabilities %.2f GB"
                         % (a_bytes / 1e9, c_bytes / 1e9)},
        "packed_tokens_per_s": M * value,
        "accepted_tokens_per_step": int(acc_len.sum() + wl.B),
        "mean_window": float(windows.mean()),
        "roofline": roof,
        "kernels": {
            "verify_attn": {"us": attn_us, "GB/s": attn_gbs, "frac_hbm": attn_gbs / hbm,
                            "TFLOP/s": attn_tfs, "frac_tensor": attn_tfs / tf_peak,
                            "bytes": a_bytes},
            "accept": {"us": accept_us, "GB/s": acc_gbs, "frac_hbm": acc_gbs / hbm,
                       "bytes": c_bytes,
                       "traffic": load_traffic("accept", wl.name, ACCEPT_SRC)},
        },
        "e2e": e2e,
        "gpu_launches": KERNELS_PER_STEP * args.steps,
        "clocks": clk.summary(),
    }
    if mode == W.MODE_CAP_ACCEPT:
        cap = step.cap_len.cpu().numpy()
        result["commit_over_cap"] = float(acc_len.sum() / max(1, cap.sum()))
    return result, inp


def sweep_arm(args, dist, world, rank, device):
    """Step rate over the batch sizes of the budget/tier sweep (Qwen3-8B shape, gamma 16,
    ctx 2048, confidence mean 0.85, cost slope 0.19 ms/token) in the three modes.
    Points whose inputs fit in L2 are marked: their per-kernel fractions are not HBM
    figures."""
    import copy
    sargs = copy.copy(args)
    sargs.steps = min(args.steps, 300)
    sargs.warmup = max(3, min(args.warmup, 20))
    sargs.kernel_iters = min(args.kernel_iters, 5)
    pts = []
    for B in W.SWEEP_B:
        for mname in ("compact", "static", "cap_accept"):
            wl = W.sweep_point(B, 0.85, 0.19)
            sargs.mode = mname
            try:
                res, inp = gpu_arm(sargs, wl, W.MODE_NAMES[mname], dist, world, rank, device,
                                   with_e2e=False)
            except RuntimeError as e:  # reported in the line, the other points still run
                pts.append({"B": B, "mode": mname, "error": str(e)})
                torch.cuda.empty_cache()
                continue
            k = res["kernels"]
            pt = {"B": B, "mode": mname, "steps_per_s": res["value"],
                  "ms_per_step": res["ms_per_step"],
                  "packed_tokens_per_s": res["packed_tokens_per_s"],
                  "accepted_tokens_per_step": res["accepted_tokens_per_step"],
                  "M": res["config"]["packed_rows_M"], "tier": res["config"]["tier"],
                  "attn_us": k["verify_attn"]["us"], "attn_frac_hbm": k["verify_attn"]["frac_hbm"],
                  "accept_us": k["accept"]["us"], "accept_frac_hbm": k["accept"]["frac_hbm"],
                  "l2_resident": k["verify_attn"]["bytes"] + k["accept"]["bytes"] < 129e6}
            if "commit_over_cap" in res:
                pt["commit_over_cap"] = res["commit_over_cap"]
            pts.append(pt)
            del inp
            torch.cuda.empty_cache()
    return pts


def e2e_arm(args, wl, mode, d, step, small, stream):
    """Same step through the public API with the per-step inputs in pinned host
    memory: H2D copies of the step's inputs, the five calls, D2H of the results,
    all inside the timed region."""
    tier = int(step.tier.item())
    row_keys = ["p_target", "q", "k_new"] + (["v_new"] if d.get("v_new") is not None else [])
    in_keys = ["conf", "draft_tok", "uniforms", "exp_noise", "p_draft"] + row_keys
    # per-row inputs: the tier's rows, as the target forward would hand them over
    dev_view = {k: (d[k][:tier] if k in row_keys else d[k]) for k in in_keys}
    host = {k: v.cpu().pin_memory() for k, v in dev_view.items()}
    out_keys = ["windows", "accept_len", "out_tok", "cstar", "committed", "n_committed"]
    host_out = {k: torch.empty_like(getattr(step, k), device="cpu").pin_memory() for k in out_keys}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())

    def one():
        for k, v in host.items():
            dev_view[k].copy_(v, non_blocking=True)
        for dst, src in small:
            dst.copy_(src, non_blocking=True)
        step.run(d, mode)
        for k in out_keys:
            host_out[k].copy_(getattr(step, k), non_blocking=True)

    n = max(3, min(args.steps, 20))
    with torch.cuda.stream(stream):
        for _ in range(2):
            one()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(n):
            one()
        b.record(stream)
    b.synchronize()
    ms = a.elapsed_time(b) / n
    return {"value": 1e3 / ms, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms, "steps": n}


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


def src_hash(paths):
    h = hashlib.sha256()
    for path in paths:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic(kernel, workload, src):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on the
    current source of the kernel."""
    p = os.path.join(PROFILES, "traffic.json")
    try:
        with open(p) as f:
            t = json.load(f)
        e = t[f"{kernel}/{workload}"]
        if e.get("src_sha256_16") == src_hash(src):
            return e["dram_bytes_per_launch"]
    except (OSError, KeyError, ValueError):
        pass
    return None


# ------------------------------------------------------------------ oracle (CPU baseline)

def oracle_sample(inp_np, wl, mode, reqs):
    """One bounded sample of the step on the CPU oracle: the global schedule and
    pack over the whole batch, then attention, acceptance and compaction for the
    sampled requests only.  Returns (seconds global, seconds for the sample)."""
    from oracle import dspark_oracle as O
    t0 = time.perf_counter()
    sch = O.schedule(inp_np["conf"], inp_np["conf_is_logit"], inp_np["sts_temp"],
                     inp_np["cost_table"], wl.max_tokens, mode)
    pk = O.pack(sch.windows, inp_np["ctx_len"], inp_np["anchor"], inp_np["draft_tok"],
                inp_np["tiers"], mode, wl.gamma)
    t1 = time.perf_counter()
    P = wl.page_size
    for r in reqs:
        c0, c1 = int(pk.cu_seqlens[r]), int(pk.cu_seqlens[r + 1])
        n = c1 - c0
        ctx = int(inp_np["ctx_len"][r])
        sub_cu = np.array([0, n])
        q = inp_np["q_dense"][r, :n]
        kn = inp_np["k_new_dense"][r, :n]
        if wl.attn == "gqa":
            O.verify_attention_gqa(q, kn, inp_np["v_new_dense"][r, :n], inp_np["k_cache"],
                                   inp_np["v_cache"], inp_np["page_table"][r:r + 1],
                                   np.array([ctx]), sub_cu, wl.Hq, wl.Hkv, 1 / math.sqrt(wl.d_qk))
        else:
            O.verify_attention_mla(q, kn, inp_np["k_cache"], inp_np["page_table"][r:r + 1],
                                   np.array([ctx]), sub_cu, wl.d_v, 1 / math.sqrt(wl.d_qk))
        pt = inp_np["p_target_dense"][r, :n]
        O.accept(pt, inp_np["p_draft"][r:r + 1], inp_np["draft_tok"][r:r + 1],
                 inp_np["uniforms"][r:r + 1], inp_np["exp_noise"][r:r + 1], sch.windows[r:r + 1],
                 sub_cu, mode, wl.gamma)
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1


def oracle_inputs(inp, reqs):
    """Host copies of what the sampled oracle step reads (only the sampled
    requests' pages of the cache, relabelled)."""
    wl = inp["workload"]
    P = wl.page_size
    out = {}
    for k in ("conf", "sts_temp", "cost_table", "tiers", "ctx_len", "anchor", "draft_tok",
              "uniforms"):
        out[k] = inp[k].cpu().numpy()
    out["conf_is_logit"] = inp["conf_is_logit"]
    B = wl.B
    pt = np.full((B, inp["page_table"].shape[1]), -1, np.int64)
    pages, k = [], 0
    for r in reqs:
        n = (int(inp["ctx_len"][r]) + P - 1) // P
        pages.append(inp["page_table"][r, :n].long())
        pt[r, :n] = np.arange(k, k + n)
        k += n
    pages = torch.cat(pages) if pages else torch.zeros(0, dtype=torch.long)
    if len(pages) == 0:
        pages = torch.zeros(1, dtype=torch.long, device=inp["k_cache"].device)
    out["page_table"] = pt
    out["k_cache"] = inp["k_cache"][pages.to(inp["k_cache"].device)].float().cpu().numpy()
    out["v_cache"] = (inp["v_cache"][pages.to(inp["v_cache"].device)].float().cpu().numpy()
                      if inp.get("v_cache") is not None else None)
    idx = torch.tensor(list(reqs), device=inp["q_dense"].device)
    for k in ("q_dense", "k_new_dense", "v_new_dense", "p_target_dense", "p_draft", "exp_noise"):
        if inp.get(k) is None:
            out[k] = None
            continue
        full = torch.zeros((B,) + tuple(inp[k].shape[1:]), dtype=torch.float32)
        full[idx.cpu()] = inp[k][idx].float().cpu()
        out[k] = full.numpy()
    out["uniforms"] = inp["uniforms"].cpu().numpy()
    return out


def oracle_timing(inp, wl, mode, budget_s, n_req):
    reqs = list(range(0, wl.B, max(1, wl.B // n_req)))[:n_req]
    inp_np = oracle_inputs(inp, reqs)
    t_glob, t_req, reps = 0.0, 0.0, 0
    t_start = time.perf_counter()
    while reps < 1 or (time.perf_counter() - t_start < budget_s and reps < 50):
        g, s = oracle_sample(inp_np, wl, mode, reqs)
        t_glob += g
        t_req += s
        reps += 1
    t_step = t_glob / reps + (t_req / reps) * wl.B / len(reqs)
    return t_step, reps, reqs


def cpu_baseline_block(t_step, reps, reqs, wl):
    return {"value": 1.0 / t_step, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": (f"{reps} x (global schedule+pack over all {wl.B} requests + attention, "
                       f"acceptance for requests {reqs}); per-request time scaled x{wl.B}/"
                       f"{len(reqs)}; numpy, one thread")}


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="dspark", choices=["dspark", "reference"])
    ap.add_argument("--workload", default="qwen3_8b", choices=sorted(W.WORKLOADS))
    ap.add_argument("--mode", default="compact", choices=list(W.MODE_NAMES))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--kernel-iters", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--sweep", action="store_true",
                    help="also report the step rate at B = 1..256 in the three modes")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world, rank, local = dist_env()
    wl = W.WORKLOADS[args.workload]
    mode = W.MODE_NAMES[args.mode]

    if args.impl == "reference":
        # the reference arm is the CPU oracle itself, on rank 0 only
        if rank != 0:
            return
        inp = W.make_inputs(wl, seed=args.seed, device="cpu")
        per = []
        n_req = 1
        reqs = list(range(0, wl.B, max(1, wl.B // n_req)))[:n_req]
        inp_np = oracle_inputs(inp, reqs)
        # Each step is one bounded sample (the global schedule + pack, and one
        # request's attention and acceptance scaled to the batch).  The oracle is
        # slow, so the run stops after ~3 minutes of samples; "steps" reports
        # how many were timed.
        t0 = time.perf_counter()
        oracle_sample(inp_np, wl, mode, reqs)
        t_one = time.perf_counter() - t0
        warm = min(args.warmup, max(1, int(20.0 / max(t_one, 1e-6))))
        n_steps = min(args.steps, max(3, int(150.0 / max(t_one, 1e-6))))
        for _ in range(warm):
            oracle_sample(inp_np, wl, mode, reqs)
        for _ in range(n_steps):
            g, s = oracle_sample(inp_np, wl, mode, reqs)
            per.append(g + s * wl.B / len(reqs))
        t_step = sum(per) / len(per)
        v = 1.0 / t_step
        line = {
            "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
            "steps": n_steps, "steps_requested": args.steps, "warmup": warm,
            "ms_per_step": t_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": workload_desc(wl, args.mode), "mode": args.mode,
                       "global_batch": wl.B, "parallelism": "cpu oracle, one thread"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": (f"each step: global schedule+pack over {wl.B} requests + "
                                        f"attention/acceptance for requests {reqs}, per-request "
                                        f"time scaled x{wl.B}/{len(reqs)}")},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line), flush=True)
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (GB300, sm_103a)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    import __graft_entry__ as g
    g.build()
    result, inp = gpu_arm(args, wl, mode, dist, world, rank, device)
    if args.sweep:
        result["sweep"] = sweep_arm(args, dist, world, rank, device)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t_step, reps, reqs = oracle_timing(inp, wl, mode, args.cpu_budget_s, 2)
        result["cpu_baseline"] = cpu_baseline_block(t_step, reps, reqs, wl)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

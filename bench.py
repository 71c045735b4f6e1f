"""Benchmark of the DSpark confidence-scheduled ragged verification step on GB300.

Headline: the Qwen3-8B-shaped workload (B=32, gamma=8, 32/8 heads x 128, context
U[1024,4096], page 16, vocab 151936 fp32 probabilities, compact mode) on one GPU.
One step = schedule -> pack -> verify attention -> accept -> compact over one
batch, captured once in a CUDA graph and replayed; the small mutable state
(page table, ctx_len, anchor, free-stack top) is restored inside the step so
that every step does identical work.

The same run also measures (keys of the one JSON line): the B=256 mixed-traffic
workload in its three modes and the latent-KV (MLA) workload (``workloads``), and
the budget/tier sweep over B x confidence mean x cost slope x mode (``sweep``), the
calibration tooling (``calibration``) and the Markov-head draft sampler at the
Qwen3-8B vocabulary (``markov_draft``); ``--no-extra`` skips them.  The CPU oracle is timed on complete steps, on one
core and on all the host's cores (``cpu_baseline``).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload qwen3_8b|mixed256|mla|tiny] [--mode compact|static|cap_accept]
                    [--no-extra] [--no-cpu-baseline] [--markov-only]

Prints one JSON line (rank 0).
"""
from __future__ import annotations

import os

# The CPU oracle (baseline leg and reference arm) runs single-threaded.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import hashlib
import re
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


def query_tile(wl, hint):
    """The attention launch a block-rows hint selects: the GQA query tile (32, 64 or 128
    columns for `hint` block rows of G heads, as the library picks it) or the latent-KV
    kernel's one tile.  A label that keys a committed DRAM-traffic figure to the launch
    configuration it was captured on."""
    if wl.attn == "mla":
        return "mla"
    rows = (wl.Hq // wl.Hkv) * max(int(hint), 1)
    return f"nt{32 if rows <= 32 else (64 if rows <= 64 else 128)}"


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
                 "--format=csv,noheader,nounits", "-lms", "50"],
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


class StepRunner:
    """One workload's inputs on the device, its VerifyStep, and one step captured in
    a CUDA graph (the small mutable state is restored inside the graph, so every
    replay does identical work)."""

    def __init__(self, inp, mode):
        import harness
        self.wl, self.mode = inp["workload"], mode
        self.d, self.step = harness.prepare(inp, mode)
        self.ctx0 = self.d["ctx_len"].cpu().numpy()
        self.small = restore_pairs(self.d, ("page_table", "ctx_len", "anchor", "free_top"))
        self.stream = torch.cuda.Stream()
        # inputs, packed rows and the state copies were made on the default stream
        self.stream.wait_stream(torch.cuda.current_stream())
        torch.cuda.synchronize()
        with torch.cuda.stream(self.stream):
            for _ in range(2):  # eager warm-up (all kernels are precompiled)
                self.one_step()
        torch.cuda.synchronize()
        check_device_error("warm-up")
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            self.one_step()
        torch.cuda.synchronize()
        st = self.step
        self.windows = st.windows.cpu().numpy()
        self.cu = st.cu_seqlens.cpu().numpy()
        self.n_rows = np.diff(self.cu)
        self.M = int(self.cu[-1])
        self.tier = int(st.tier.item())

    def one_step(self):
        for dst, src in self.small:
            dst.copy_(src, non_blocking=True)
        self.step.run(self.d, self.mode)

    def replay(self, n):
        with torch.cuda.stream(self.stream):
            for _ in range(n):
                self.graph.replay()

    def time_replays(self, n, dist=None, device=None):
        """Device time (ms) of n graph replays between CUDA events on the launching
        stream, with a barrier and synchronize on both sides."""
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(dist, device or torch.device("cuda"))
        with torch.cuda.stream(self.stream):
            ev0.record(self.stream)
            for _ in range(n):
                self.graph.replay()
            ev1.record(self.stream)
        ev1.synchronize()
        barrier(dist, device or torch.device("cuda"))
        return ev0.elapsed_time(ev1)

    def steps_for(self, seconds, lo=30, hi=2000):
        """Replays that fill about `seconds` of device time (bounded)."""
        ms = self.time_replays(5) / 5
        return int(min(hi, max(lo, seconds * 1e3 / max(ms, 1e-3))))

    def time_call(self, fn, reps, iters):
        """us per call of fn, from a graph of `reps` back-to-back calls replayed
        `iters` times between CUDA events on the launching stream."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            for _ in range(reps):
                fn()
        with torch.cuda.stream(self.stream):
            for _ in range(2):
                g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            a.record(self.stream)
            for _ in range(iters):
                g.replay()
            b.record(self.stream)
        b.synchronize()
        return a.elapsed_time(b) * 1e3 / (reps * iters)

    def kernel_figures(self, iters, reps=10):
        """The step's attention call (over the work list its own pack call built, from
        the restored state) and its acceptance call, each timed alone; algorithmic
        bytes, flops and roofline fractions."""
        st, d, wl = self.step, self.d, self.wl
        with torch.cuda.stream(self.stream):
            for dst, src in self.small:
                dst.copy_(src, non_blocking=True)
            st.pack_plan(d, self.mode)
        torch.cuda.synchronize()
        attn_us = self.time_call(lambda: st.attention_planned(d), reps, iters)
        accept_us = self.time_call(lambda: st.accept(d, self.mode), reps, iters)
        check_device_error("per-call timing")
        acc_len = st.accept_len.cpu().numpy()
        a_bytes = attn_bytes(wl, self.ctx0, self.n_rows)
        a_flops = attn_flops(wl, self.ctx0, self.n_rows)
        c_bytes = accept_bytes(wl, self.windows, self.n_rows, acc_len, self.mode)
        peaks = peak_values()
        attn_gbs = a_bytes / (attn_us * 1e-6) / 1e9
        attn_tfs = a_flops / (attn_us * 1e-6) / 1e12
        acc_gbs = c_bytes / (accept_us * 1e-6) / 1e9
        return {
            "verify_attn": {"us": attn_us, "GB/s": attn_gbs, "frac_hbm": attn_gbs / peaks["hbm"],
                            "TFLOP/s": attn_tfs, "frac_tensor": attn_tfs / peaks["tf"],
                            "bytes": a_bytes, "flops": a_flops,
                            "launch": query_tile(wl, st.block_rows_hint)},
            "accept": {"us": accept_us, "GB/s": acc_gbs, "frac_hbm": acc_gbs / peaks["hbm"],
                       "bytes": c_bytes},
        }

    def time_step_graph(self, n):
        """The same step as the library's own step graph (tier chosen on the device by a
        switch node; dspark_step_graph_*), launched n times back to back on the stream,
        each launch preceded by the copy that restores the small mutable state: two
        stream operations per step and no host synchronisation between steps.  Returns
        (ms for the n steps, step rate)."""
        g = self.step.graph(self.d, self.mode)
        try:
            def one():
                for dst, src in self.small:
                    dst.copy_(src, non_blocking=True)
                g.launch(self.stream)
            with torch.cuda.stream(self.stream):
                for _ in range(5):
                    one()
            torch.cuda.synchronize()
            check_device_error("step graph warm-up")
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(self.stream):
                a.record(self.stream)
                for _ in range(n):
                    one()
                b.record(self.stream)
            b.synchronize()
            check_device_error("step graph")
            ms = a.elapsed_time(b)
            self.step_graph_pdl = g.pdl
        finally:
            g.close()
        return ms, n / (ms / 1e3)

    def outcome(self):
        """Accepted tokens of the step (committed drafts + one bonus/correction per
        request) and, in cap-accept mode, the commit/cap utilisation."""
        acc = self.step.accept_len.cpu().numpy()
        out = {"accepted_tokens_per_step": int(acc.sum() + self.wl.B),
               "mean_window": float(self.windows.mean())}
        if self.mode == W.MODE_CAP_ACCEPT:
            cap = self.step.cap_len.cpu().numpy()
            out["commit_over_cap"] = float(acc.sum() / max(1, cap.sum()))
        return out


def check_device_error(where):
    import speculative_decoding_verification_dspark_gb300 as dspark
    err = dspark.read_device_error()
    if err:
        raise RuntimeError(f"device error word {err:#x} ({where})")


def peak_values():
    peaks = load_peaks()
    hbm, tf = peaks.get("hbm_gbs"), peaks.get("bf16_tflops")
    return {"hbm": hbm or 6800.0, "hbm_src": "measured" if hbm else "fallback",
            "tf": tf or 1900.0, "tf_src": "measured" if tf else "fallback"}


def roofline_block(wl, kf):
    """The dominant kernel's roofline: the attention call, HBM-bound unless its flops
    per algorithmic byte exceed the ridge point of the measured peaks."""
    pk = peak_values()
    a = kf["verify_attn"]
    traffic = load_traffic("verify_attn", wl.name, attn_src(wl), a.get("launch"))
    common = {"kernel": "dspark_verify_attn (main kernel + combine; work list from the pack call)",
              "launch": a.get("launch"), "traffic": traffic, "algorithmic_bytes": a["bytes"], "us_per_launch": a["us"]}
    if a["flops"] / max(a["bytes"], 1) > pk["tf"] * 1e12 / (pk["hbm"] * 1e9):
        return {"bound": "tensor", "achieved": a["TFLOP/s"], "peak": pk["tf"], "unit": "TFLOP/s",
                "frac": a["TFLOP/s"] / pk["tf"], "algorithmic_flops": a["flops"], **common,
                "peak_source": f"{pk['tf_src']} bf16_tflops (burst cuBLAS GEMM; the call is "
                               "timed alone)"}
    return {"bound": "hbm", "achieved": a["GB/s"], "peak": pk["hbm"], "unit": "GB/s",
            "frac": a["GB/s"] / pk["hbm"], **common,
            "peak_source": f"{pk['hbm_src']} hbm_gbs (burst copy)"}


def gpu_arm(args, wl, mode, dist, world, rank, device, with_e2e=True):
    """The headline: timed graph replays of the step, per-call kernel figures, the
    end-to-end leg through the public API with host buffers, and the clocks sampled
    over the whole busy window (warm-up, timed steps, per-call timing)."""
    inp = W.make_inputs(wl, seed=args.seed + rank, device=W.gen_device(wl))
    run = StepRunner(inp, mode)
    with ClockSampler(device.index or 0) as clk:
        # warm-up: W replays at least, and at least ~0.5 s of device time so that the
        # clock record has samples under load before the timed region
        n_warm = max(args.warmup, run.steps_for(0.5))
        run.replay(n_warm)
        torch.cuda.synchronize()
        ms = run.time_replays(args.steps, dist, device)
        ms_max = max_over_ranks(ms, dist, device)
        check_device_error("timed region")
        kf = run.kernel_figures(args.kernel_iters)
    kf["accept"]["traffic"] = load_traffic("accept", wl.name, ACCEPT_SRC)
    sg_ms, sg_rate = run.time_step_graph(max(args.steps, 200))
    e2e = e2e_arm(args, run) if with_e2e else None
    check_device_error("end-to-end leg")
    value = world * args.steps / (ms_max / 1e3)
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "dtype_detail": "attention bf16 operands / fp32 accumulate and softmax; acceptance fp32",
        "data": "synthetic",
        "config": {"workload": workload_desc(wl, args.mode), "mode": args.mode,
                   "global_batch": wl.B * world, "packed_rows_M": run.M, "tier": run.tier,
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (no flush): KV %.2f GB, probabilities %.2f GB"
                         % (kf["verify_attn"]["bytes"] / 1e9, kf["accept"]["bytes"] / 1e9)},
        "packed_tokens_per_s": run.M * value,
        **run.outcome(),
        "roofline": roofline_block(wl, kf),
        "kernels": kf,
        "e2e": e2e,
        "step_graph": {"steps_per_s": sg_rate, "ms_per_step": sg_ms / max(args.steps, 200),
                       "steps": max(args.steps, 200), "pdl": run.step_graph_pdl,
                       "what": "the library's step graph (tier chosen on the device by a switch "
                               "node), launched back to back after the state-restore copy: "
                               "two host launches per step, no host synchronisation"},
        "gpu_launches": KERNELS_PER_STEP * args.steps,
        "clocks": {**clk.summary(), "window": "warm-up (>= 0.5 s), timed steps and per-call "
                                              "timing of the headline"},
    }
    del run
    torch.cuda.empty_cache()
    return result, inp


def point_figures(run, seconds=0.15, kernel_iters=3):
    """Step rate and per-call figures of one extra workload point."""
    n = run.steps_for(seconds)
    run.replay(3)
    ms = run.time_replays(n)
    check_device_error("extra point")
    kf = run.kernel_figures(kernel_iters, reps=5)
    run.last_kernels = kf
    sps = n / (ms / 1e3)
    pt = {"steps_per_s": sps, "ms_per_step": ms / n, "steps_timed": n, "M": run.M,
          "tier": run.tier, "packed_tokens_per_s": run.M * sps, **run.outcome(),
          "attn_us": kf["verify_attn"]["us"], "attn_frac_hbm": kf["verify_attn"]["frac_hbm"],
          "attn_frac_tensor": kf["verify_attn"]["frac_tensor"],
          "accept_us": kf["accept"]["us"], "accept_frac_hbm": kf["accept"]["frac_hbm"],
          "l2_resident": kf["verify_attn"]["bytes"] + kf["accept"]["bytes"] < 129e6}
    return pt


def workloads_arm(seed):
    """The other full-size workloads: mixed traffic at B=256 in its three modes, and
    the latent-KV shape, each a CUDA-graph step timed like the headline."""
    out = {}
    for name, modes in (("mixed256", ("compact", "static", "cap_accept")), ("mla", ("compact",))):
        wl = W.WORKLOADS[name]
        inp = W.make_inputs(wl, seed=seed, device=W.gen_device(wl))
        out[name] = {"workload": workload_desc(wl, "/".join(modes))}
        for mname in modes:
            run = StepRunner(inp, W.MODE_NAMES[mname])
            pt = point_figures(run, seconds=0.3, kernel_iters=5)
            pt["roofline"] = roofline_block(wl, run.last_kernels)
            out[name][mname] = pt
            del run
            torch.cuda.empty_cache()
        del inp
        torch.cuda.empty_cache()
    return out


def sweep_arm(seed):
    """The budget/tier sweep: B in {1, 8, 32, 128, 256} x confidence mean in
    {.95, .85, .70} x cost slope in {.05, .19, .5} ms/token (Qwen3-8B heads,
    gamma 16, ctx 2048, tiers 4..4096), compact and cap-accept at every point;
    static verifies the whole block whatever the slope, so it is timed once per
    (B, confidence).  Inputs are drawn once per (B, confidence); the slope changes
    only the cost table.  Points whose inputs fit in L2 are marked."""
    pts = []
    for B in W.SWEEP_B:
        for c in W.SWEEP_CONF_MEANS:
            base = W.make_inputs(W.sweep_point(B, c, W.SWEEP_THETA[0]), seed,
                                 device=W.gen_device(W.sweep_point(B, c, 0.19)))
            for theta in W.SWEEP_THETA:
                wl = W.sweep_point(B, c, theta)
                m = torch.arange(base["cost_table"].numel(), dtype=torch.float64,
                                 device=base["cost_table"].device)
                inp = dict(base, workload=wl,
                           cost_table=(wl.cost_bias_ms + theta * m).to(torch.float32))
                modes = ("compact", "cap_accept") + (("static",) if theta == 0.19 else ())
                for mname in modes:
                    try:
                        run = StepRunner(inp, W.MODE_NAMES[mname])
                        pt = point_figures(run)
                        del run
                    except RuntimeError as e:  # reported in the line; the others still run
                        pt = {"error": str(e)}
                    pts.append({"B": B, "conf_mean": c,
                                "theta_ms": theta if mname != "static" else "any",
                                "mode": mname, **pt})
                    torch.cuda.empty_cache()
            del base
            torch.cuda.empty_cache()
    return pts


def calib_arm(seed):
    """Calibration tooling at a serving-sized store: B = 1024 requests, gamma = 8, one
    collect per step (cap-accept outcomes, every position labelled) until 2^17
    samples per position, then the ECE (15 bins) and the STS refit (36 bisections)
    over the full store.  Times: collect per call (a graph of calls), ECE and refit
    per call."""
    import speculative_decoding_verification_dspark_gb300 as dspark
    dev = torch.device("cuda")
    B, gamma, cap = 1024, 8, 1 << 17
    g = torch.Generator(device=dev).manual_seed(seed * 7919 + 17)
    c = 0.6 + 0.4 * torch.rand((B, gamma), generator=g, device=dev)
    a = torch.cumprod(c, dim=1).float().contiguous()          # synthetic survival input
    a_hat = (a * 0.9).contiguous()
    windows = torch.full((B,), gamma, dtype=torch.int32, device=dev)
    cap_len = torch.randint(0, gamma + 1, (B,), generator=g, device=dev, dtype=torch.int32)
    store = dspark.CalibStore(gamma, cap)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    calls = cap // B
    reps = 8
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(reps):
            store.collect(a, a_hat, windows, cap_len, W.MODE_CAP_ACCEPT)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    with torch.cuda.stream(stream):
        store.count.zero_()
        ev[0].record(stream)
        for _ in range(calls // reps):
            graph.replay()
        ev[1].record(stream)
        ev[2].record(stream)
        store.ece(15)
        ev[3].record(stream)
        ev[4].record(stream)
        store.sts_fit(36)
        ev[5].record(stream)
    ev[5].synchronize()
    check_device_error("calibration")
    n = int(store.count.min().item())
    return {"requests_per_collect": B, "gamma": gamma, "samples_per_position": n,
            "collect_us": ev[0].elapsed_time(ev[1]) * 1e3 / calls,
            "ece_ms": ev[2].elapsed_time(ev[3]), "sts_fit_ms": ev[4].elapsed_time(ev[5]),
            "sts_fit_bisections": 36, "ece_bins": 15}


MARKOV_SRC = [os.path.join(_CSRC, f) for f in ("markov_draft.cu", "ptx.cuh", "common.cuh")]


def markov_bytes(B, gamma, V, rank=256):
    """Algorithmic bytes of one draft block: W2 read once, the base logits U and the
    noise read once, p written once, the W1 rows of the B*gamma conditioning tokens,
    the anchors and the tokens."""
    return rank * V * 2 + 3 * B * gamma * V * 4 + B * gamma * rank * 2 + B * 4 + B * gamma * 4


def markov_arm(seed, reps=20, oracle_rows=2, with_oracle=True):
    """Markov-head draft sampling of one block (dspark_markov_draft) at the Qwen3-8B
    vocabulary with the verification workload's batch and block (B = 32, gamma = 8,
    V = 151936, rank 256): device time per block with L2 flushed before each call,
    its HBM roofline, and the oracle timed on `oracle_rows` request rows (fp64)."""
    import speculative_decoding_verification_dspark_gb300 as dspark
    cfg = W.MARKOV_WORKLOADS["markov_qwen3_8b"]
    B, gamma, V = cfg["B"], cfg["gamma"], cfg["V"]
    inp = W.make_markov_inputs(B, gamma, V, seed=seed, device="cuda")
    md = dspark.MarkovDraft(V)
    tok = torch.empty(B, gamma, dtype=torch.int32, device="cuda")
    p = torch.empty(B, gamma, V, dtype=torch.float32, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    args = (inp["U"], inp["W1"], inp["W2"], inp["anchor"], inp["exp_noise"], tok, p)
    for _ in range(3):
        md(*args)
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        md(*args)
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b) * 1e3)
    check_device_error("markov draft")
    us = statistics.median(ts)
    nbytes = markov_bytes(B, gamma, V)
    pk = peak_values()
    gbs = nbytes / (us * 1e-6) / 1e9
    t_row = None
    if with_oracle:
        # the oracle (CPU baseline leg): the same block for a few request rows
        from oracle import dspark_oracle as O
        rows = slice(0, oracle_rows)
        U = inp["U"][rows].cpu().numpy()
        W1 = inp["W1"].float().cpu().numpy()
        W2 = inp["W2"].float().cpu().numpy()
        e = inp["exp_noise"][rows].cpu().numpy()
        anc = inp["anchor"][rows].cpu().numpy()
        t0 = time.perf_counter()
        O.markov_draft(U, W1, W2, anc, e)
        t_row = (time.perf_counter() - t0) / oracle_rows
    del inp, p, flush
    torch.cuda.empty_cache()
    return {"workload": f"Markov-head draft block: B={B}, gamma={gamma}, V={V}, rank 256, "
                        "fp32 U and noise, bf16 W1/W2 (random weights)",
            "us_per_block": us, "us_min": min(ts), "blocks_per_s": 1e6 / us,
            "draft_tokens_per_s": B * gamma * 1e6 / us, "launches_per_block": -(-B // 32),
            "l2": "flushed before each call (256 MB written)",
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm"], "unit": "GB/s",
                         "frac": gbs / pk["hbm"], "algorithmic_bytes": nbytes,
                         "traffic": load_traffic("markov_draft", "markov_qwen3_8b", MARKOV_SRC),
                         "peak_source": f"{pk['hbm_src']} hbm_gbs (burst copy)"},
            "cpu_oracle": None if t_row is None else {
                "blocks_per_s": 1.0 / (t_row * B), "cores": 1, "kind": "oracle",
                "sample": f"{oracle_rows} request rows of the block (fp64), scaled to {B} rows"}}


def e2e_arm(args, run):
    """The same step through the public API with the step's inputs in pinned host
    memory: host-to-device copies of the inputs (the M packed rows of the per-row
    tensors, as the target forward hands them over, and the per-request tensors),
    the five calls, and the device-to-host copy of the results, all inside the
    timed region."""
    d, step, M = run.d, run.step, run.M
    row_keys = ["p_target", "q", "k_new"] + (["v_new"] if d.get("v_new") is not None else [])
    in_keys = ["conf", "draft_tok", "uniforms", "exp_noise", "p_draft"] + row_keys
    dev_view = {k: (d[k][:M] if k in row_keys else d[k]) for k in in_keys}
    host = {k: v.cpu().pin_memory() for k, v in dev_view.items()}
    out_keys = ["windows", "accept_len", "out_tok", "cstar", "committed", "n_committed"]
    host_out = {k: torch.empty_like(getattr(step, k), device="cpu").pin_memory() for k in out_keys}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())

    def one():
        for k, v in host.items():
            dev_view[k].copy_(v, non_blocking=True)
        for dst, src in run.small:
            dst.copy_(src, non_blocking=True)
        step.run(d, run.mode)
        for k in out_keys:
            host_out[k].copy_(getattr(step, k), non_blocking=True)

    n = max(3, min(args.steps, 20))
    stream = run.stream
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


_COMMENT = re.compile(r"//[^\n]*|/\*.*?\*/", re.S)


def src_hash(paths):
    """Hash of the sources' code: comments and whitespace left out, so that a change
    of wording alone keeps a capture taken on the same code."""
    h = hashlib.sha256()
    for path in paths:
        with open(path, encoding="utf-8") as f:
            code = _COMMENT.sub(" ", f.read())
        h.update(" ".join(code.split()).encode())
    return h.hexdigest()[:16]


def load_traffic(kernel, workload, src, launch=None):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on the
    current source of the kernel (and, for the attention, on the same launch
    configuration)."""
    p = os.path.join(PROFILES, "traffic.json")
    try:
        with open(p) as f:
            t = json.load(f)
        e = t[f"{kernel}/{workload}"]
        if e.get("src_sha256_16") == src_hash(src) and e.get("launch") == launch:
            return e["dram_bytes_per_launch"]
    except (OSError, KeyError, ValueError):
        pass
    return None


# ------------------------------------------------------------------ oracle (CPU baseline)
#
# The oracle times complete steps: the global schedule and pack, the attention of
# every request, the acceptance of every request, and the compaction of the batch,
# each by the oracle's own functions as they stand.  The per-request attention and
# acceptance run either one after another in this process (one core) or spread
# over a pool of worker processes, one per host core (all cores).  The workers read
# the step's inputs from memory-mapped files written once before the timing (the
# inputs as the target forward would hand them over), so no input is copied
# between processes inside the timed region.

_OW = {}  # worker-side: the memory-mapped inputs of the step


def _oracle_worker_init(folder, meta):
    import numpy as _np
    _OW.clear()
    _OW["meta"] = meta
    for k, (shape, dtype) in meta["arrays"].items():
        _OW[k] = _np.memmap(os.path.join(folder, k + ".bin"), dtype=dtype, mode="r",
                            shape=tuple(shape))


def _oracle_request(task):
    """Attention and acceptance of one request by the oracle's functions."""
    from oracle import dspark_oracle as O
    r, c0, c1, w_r = task
    m = _OW["meta"]
    a = _OW
    sub_cu = np.array([0, c1 - c0])
    ctx = a["ctx_len"][r:r + 1]
    if m["attn"] == "gqa":
        o, lse = O.verify_attention_gqa(a["q"][c0:c1], a["k_new"][c0:c1], a["v_new"][c0:c1],
                                        a["k_cache"], a["v_cache"], a["page_table"][r:r + 1], ctx,
                                        sub_cu, m["Hq"], m["Hkv"], m["scale"])
    else:
        o, lse = O.verify_attention_mla(a["q"][c0:c1], a["k_new"][c0:c1], a["k_cache"],
                                        a["page_table"][r:r + 1], ctx, sub_cu, m["d_v"],
                                        m["scale"])
    acc = O.accept(a["p_target"][c0:c1], a["p_draft"][r:r + 1], a["draft_tok"][r:r + 1],
                   a["uniforms"][r:r + 1], a["exp_noise"][r:r + 1], np.array([w_r], np.int32),
                   sub_cu, m["mode"], m["gamma"])
    return r, float(np.sum(o)), int(acc.accept_len[0]), int(acc.out_tok[0])


class OracleBaseline:
    """Complete oracle steps of one workload on the host cores."""

    def __init__(self, inp, mode, cores=None):
        import tempfile
        from oracle import dspark_oracle as O
        wl = inp["workload"]
        self.wl, self.mode = wl, mode
        h = {k: (v.float() if v.dtype == torch.bfloat16 else v).cpu().numpy()
             for k, v in inp.items() if isinstance(v, torch.Tensor)}
        h["conf_is_logit"] = inp["conf_is_logit"]
        self.h = h
        # the packed rows the target forward hands over (laid out with the oracle's
        # own cu_seqlens, as in the GPU tests)
        sch = O.schedule(h["conf"], h["conf_is_logit"], h["sts_temp"], h["cost_table"],
                         wl.max_tokens, mode)
        pk = O.pack(sch.windows, h["ctx_len"], h["anchor"], h["draft_tok"], h["tiers"], mode,
                    wl.gamma)
        cu = torch.as_tensor(pk.cu_seqlens)
        packed = {"q": inp["q_dense"], "k_new": inp["k_new_dense"],
                  "p_target": inp["p_target_dense"]}
        if inp.get("v_new_dense") is not None:
            packed["v_new"] = inp["v_new_dense"]
        for k, v in packed.items():
            h[k] = W.to_packed(v.cpu(), cu, pk.tier).float().numpy()
        self.folder = tempfile.mkdtemp(prefix="dspark_oracle_")
        arrays = {}
        for k in ("q", "k_new", "v_new", "p_target", "k_cache", "v_cache", "page_table",
                  "ctx_len", "p_draft", "draft_tok", "uniforms", "exp_noise"):
            if h.get(k) is None:
                continue
            a = np.ascontiguousarray(h[k])
            a.tofile(os.path.join(self.folder, k + ".bin"))
            arrays[k] = (list(a.shape), a.dtype.str)
        self.meta = {"arrays": arrays, "attn": wl.attn, "Hq": wl.Hq, "Hkv": wl.Hkv,
                     "d_v": wl.d_v, "scale": 1.0 / math.sqrt(wl.d_qk), "mode": mode,
                     "gamma": wl.gamma}
        _oracle_worker_init(self.folder, self.meta)  # this process serves the one-core runs
        self.cores = cores or len(os.sched_getaffinity(0))
        self.pool = None

    def start_pool(self):
        import multiprocessing as mp
        if self.pool is None:
            ctx = mp.get_context("spawn")
            self.pool = ctx.Pool(self.cores, initializer=_oracle_worker_init,
                                 initargs=(self.folder, self.meta))
            self.pool.map(_oracle_request_noop, range(self.cores))  # workers up
        return self.pool

    def step(self, parallel):
        """One complete oracle step; returns its wall time in seconds."""
        from oracle import dspark_oracle as O
        h, wl, mode = self.h, self.wl, self.mode
        t0 = time.perf_counter()
        sch = O.schedule(h["conf"], h["conf_is_logit"], h["sts_temp"], h["cost_table"],
                         wl.max_tokens, mode)
        pk = O.pack(sch.windows, h["ctx_len"], h["anchor"], h["draft_tok"], h["tiers"], mode,
                    wl.gamma)
        tasks = [(r, int(pk.cu_seqlens[r]), int(pk.cu_seqlens[r + 1]), int(sch.windows[r]))
                 for r in range(wl.B)]
        if parallel:
            res = self.start_pool().map(_oracle_request, tasks, chunksize=1)
        else:
            res = [_oracle_request(t) for t in tasks]
        res.sort()
        L = np.array([x[2] for x in res], np.int32)
        tok = np.array([x[3] for x in res], np.int32)
        O.compact(_OW["k_new"], _OW.get("v_new"), pk.cu_seqlens, L, tok, h["draft_tok"],
                  wl.page_size, h["page_table"], h["ctx_len"], h["anchor"], h["free_pages"],
                  int(h["free_top"][0]), _OW["k_cache"], _OW.get("v_cache"))
        return time.perf_counter() - t0

    def time_steps(self, parallel, budget_s, max_steps, warmup=1):
        for _ in range(warmup):
            self.step(parallel)
        ts = []
        t_start = time.perf_counter()
        while len(ts) < max_steps and (not ts or time.perf_counter() - t_start < budget_s):
            ts.append(self.step(parallel))
        return ts

    def close(self):
        import shutil
        if self.pool is not None:
            self.pool.terminate()
            self.pool.join()
            self.pool = None
        _OW.clear()
        shutil.rmtree(self.folder, ignore_errors=True)


def _oracle_request_noop(i):
    return i


def cpu_baseline(inp, mode, budget_s):
    """The oracle as it stands on the host cores: complete steps on one core, then on
    all cores.  The all-cores figure is the line's value."""
    ob = OracleBaseline(inp, mode)
    try:
        t1 = ob.time_steps(False, budget_s / 2, 20)
        tn = ob.time_steps(True, budget_s / 2, 50)
    finally:
        ob.close()
    wl = inp["workload"]
    m1, mn = statistics.median(t1), statistics.median(tn)
    return {"value": 1.0 / mn, "unit": UNIT, "cores": ob.cores, "kind": "oracle",
            "value_1core": 1.0 / m1, "steps_timed": len(tn), "steps_timed_1core": len(t1),
            "host_cores": ob.cores,
            "sample": (f"complete steps of the {wl.name} workload (global schedule and pack, "
                       f"attention and acceptance of all {wl.B} requests, compaction of the "
                       f"batch; median of {len(tn)} steps on {ob.cores} worker processes, "
                       f"{len(t1)} steps on one core); numpy, one BLAS thread per process")}


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
    ap.add_argument("--cpu-budget-s", type=float, default=20.0)
    ap.add_argument("--no-extra", action="store_true",
                    help="time the headline only (no other workloads, no sweep)")
    ap.add_argument("--markov-only", action="store_true",
                    help="time the Markov-head draft block alone (its JSON key, one line)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world, rank, local = dist_env()
    wl = W.WORKLOADS[args.workload]
    mode = W.MODE_NAMES[args.mode]

    if args.impl == "reference":
        # the reference arm is the CPU oracle itself, on rank 0 only, on all the
        # host's cores; each step is a complete step of the workload
        if rank != 0:
            return
        inp = W.make_inputs(wl, seed=args.seed, device="cpu")
        ob = OracleBaseline(inp, mode)
        try:
            t0 = time.perf_counter()
            ob.step(True)  # also starts the worker pool
            t_one = max(time.perf_counter() - t0, 1e-6)
            # the whole run within ~3 minutes: fewer steps than asked if need be
            warm = min(args.warmup, max(1, int(20.0 / t_one)))
            n_steps = min(args.steps, max(3, int(150.0 / t_one)))
            ts = ob.time_steps(True, 1e9, n_steps, warmup=warm)
        finally:
            ob.close()
        t_step = statistics.mean(ts)
        v = 1.0 / t_step
        line = {
            "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
            "steps": len(ts), "steps_requested": args.steps, "warmup": warm,
            "ms_per_step": t_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": workload_desc(wl, args.mode), "mode": args.mode,
                       "global_batch": wl.B,
                       "parallelism": f"cpu oracle, {ob.cores} worker processes"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": ob.cores, "kind": "oracle",
                             "sample": (f"{len(ts)} complete steps (schedule, pack, attention "
                                        f"and acceptance of all {wl.B} requests, compaction) "
                                        f"on {ob.cores} worker processes")},
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
    if args.markov_only:
        if rank == 0:
            mk = markov_arm(args.seed, reps=max(args.steps, 3), with_oracle=not args.no_cpu_baseline)
            print(json.dumps({"markov_draft": mk}), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return
    result, inp = gpu_arm(args, wl, mode, dist, world, rank, device)
    # the extra workloads and the sweep: one-GPU runs only (the scaling runs time the
    # headline alone)
    if world == 1 and not args.no_extra:
        t0 = time.perf_counter()
        result["workloads"] = workloads_arm(args.seed)
        result["sweep"] = sweep_arm(args.seed)
        result["calibration"] = calib_arm(args.seed)
        result["markov_draft"] = markov_arm(args.seed)
        result["extra_wall_s"] = time.perf_counter() - t0
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(inp, mode, args.cpu_budget_s)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

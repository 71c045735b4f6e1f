"""Python binding of libdspark.so (ctypes): argument marshalling only.

Every step of the verification path runs in the library's CUDA kernels; this
module converts torch tensors to raw device pointers, passes the current CUDA
stream, and turns non-zero status codes into exceptions.  PyTorch is used for
device memory and streams only.  Importing works without a GPU; calling needs
one (sm_103a) and the built library -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "COMPACT", "STATIC", "CAP_ACCEPT", "F32", "BF16", "DSparkError", "lib", "load",
    "block_rows_hint_for",
    "schedule", "pack", "verify_attn", "accept", "accept_noalloc", "compact", "read_device_error",
    "verify_attn_workspace_size", "accept_workspace_size", "compact_workspace_size",
    "VerifyStep", "StepGraph", "CalibStore", "DEVERR",
]

COMPACT, STATIC, CAP_ACCEPT = 0, 1, 2
F32, BF16 = 0, 1
DEVERR = {
    0x1: "rows_overflow", 0x2: "no_free_page", 0x4: "page_row_full", 0x8: "wait_timeout",
    0x10: "bad_input", 0x20: "work_overflow",
}

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdspark.so")

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_Z = ctypes.c_size_t

_SIGNATURES = {
    "dspark_status_string": (ctypes.c_char_p, [_I]),
    "dspark_read_device_error": (_I, [_P]),
    "dspark_num_sms": (_I, []),
    "dspark_set_wait_limit_ns": (_I, [ctypes.c_ulonglong]),
    "dspark_set_wait_probe": (_I, [_I]),
    "dspark_schedule": (_I, [_P, _I, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "dspark_calib_collect": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _I, _P]),
    "dspark_calib_ece": (_I, [_P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P]),
    "dspark_sts_fit_workspace_size": (_Z, [_I, _I]),
    "dspark_sts_fit": (_I, [_P, _P, _P, _I, _I, _I, _P, _P, _Z, _P]),
    "dspark_block_accept_estimate": (_I, [_P, _P, _I, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                          _P, _P, _P]),
    "dspark_markov_draft_workspace_size": (_Z, [_I]),
    "dspark_markov_draft": (_I, [_P, _P, _P, _I, _P, _P, _I, _I, _I, _P, _P, _P, _Z, _P]),
    "dspark_pack": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]),
    "dspark_verify_attn_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "dspark_verify_attn": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                _F, _I, _I, _P, _P, _P, _Z, _P]),
    "dspark_verify_attn_planned": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _P, _P, _I, _I, _I, _I, _I,
                                        _I, _I, _F, _I, _I, _P, _P, _P, _Z, _P]),
    "dspark_pack_plan": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                              _I, _I, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "dspark_accept_workspace_size": (_Z, [_I, _I, _I, _I]),
    "dspark_accept": (_I, [_P, _P, _I, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P,
                           _P, _Z, _P]),
    "dspark_accept_noalloc": (_I, [_P, _P, _I, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P,
                                   _P, _P, _P]),
    "dspark_compact_workspace_size": (_Z, [_I]),
    "dspark_step_graph_create": (_I, [_P, _P]),
    "dspark_step_graph_launch": (_I, [_P, _P]),
    "dspark_step_graph_destroy": (_I, [_P]),
    "dspark_step_graph_flags": (_I, [_P]),
    "dspark_compact": (_I, [_P, _P, _I, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P,
                            _P, _P, _P, _P, _Z, _P]),
}

_lib = None


class DSparkError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = lib().dspark_status_string(status).decode()
        super().__init__(f"{fn} failed: {msg} ({status})")
        self.status = status


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the in-tree library; raise if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build it with __graft_entry__.build() "
                              "(speculative_decoding_verification_dspark_gb300/build.py)")
        l = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


lib = load


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn, rc):
    if rc != 0:
        raise DSparkError(fn, rc)


def read_device_error(stream=None) -> int:
    rc = lib().dspark_read_device_error(_stream(stream))
    if rc < 0:
        raise DSparkError("dspark_read_device_error", rc)
    return rc


def num_sms() -> int:
    return lib().dspark_num_sms()


def set_wait_limit_ns(ns: int) -> None:
    """Limit of the acceptance pass's bounded waits on the current device (0: 2 s)."""
    _check("dspark_set_wait_limit_ns", lib().dspark_set_wait_limit_ns(int(ns)))


def set_wait_probe(on: bool) -> None:
    """Test hook: the acceptance pass first waits on a barrier nothing arrives at."""
    _check("dspark_set_wait_probe", lib().dspark_set_wait_probe(1 if on else 0))


def schedule(conf, conf_is_logit, sts_temp, cost_table, max_tokens, mode, windows, a_hat, M_out,
             E_out, stream=None, survival=None):
    """``survival``: optional fp32 [B, gamma] output of the uncalibrated prefix survival."""
    B, gamma = conf.shape
    _check("dspark_schedule", lib().dspark_schedule(
        _ptr(conf), int(conf_is_logit), _ptr(sts_temp), _ptr(cost_table), cost_table.numel(), B,
        gamma, int(max_tokens), int(mode), _ptr(windows), _ptr(a_hat), _ptr(survival),
        _ptr(M_out), _ptr(E_out), _stream(stream)))


class CalibStore:
    """Device store of labelled accept outcomes per draft position (dspark_calib_*):
    ``collect`` after a step, ``ece`` and ``sts_fit`` on demand."""

    def __init__(self, gamma, capacity, device="cuda"):
        dev = torch.device(device)
        self.gamma, self.capacity = gamma, capacity
        self.s_a = torch.zeros(gamma, capacity, dtype=torch.float32, device=dev)
        self.s_ahat = torch.zeros(gamma, capacity, dtype=torch.float32, device=dev)
        self.s_y = torch.zeros(gamma, capacity, dtype=torch.int8, device=dev)
        self.count = torch.zeros(gamma, dtype=torch.int32, device=dev)
        self.ws = torch.empty(lib().dspark_sts_fit_workspace_size(gamma, capacity),
                              dtype=torch.uint8, device=dev)

    def collect(self, survival, a_hat, windows, cap_len, mode, stream=None):
        B = windows.numel()
        _check("dspark_calib_collect", lib().dspark_calib_collect(
            _ptr(survival), _ptr(a_hat), _ptr(windows), _ptr(cap_len), int(mode), B, self.gamma,
            _ptr(self.s_a), _ptr(self.s_ahat), _ptr(self.s_y), _ptr(self.count), self.capacity,
            _stream(stream)))

    def ece(self, n_bins, stream=None):
        """(ece fp64 [1], bin counts, bin sums of a_hat, bin sums of y) on the device."""
        dev = self.count.device
        bn = torch.zeros(n_bins, dtype=torch.int32, device=dev)
        bp = torch.zeros(n_bins, dtype=torch.float64, device=dev)
        by = torch.zeros(n_bins, dtype=torch.float64, device=dev)
        e = torch.zeros(1, dtype=torch.float64, device=dev)
        _check("dspark_calib_ece", lib().dspark_calib_ece(
            _ptr(self.s_ahat), _ptr(self.s_y), _ptr(self.count), self.capacity, self.gamma,
            int(n_bins), _ptr(bn), _ptr(bp), _ptr(by), _ptr(e), _stream(stream)))
        return e, bn, bp, by

    def sts_fit(self, iters, temps=None, stream=None):
        """Refitted STS temperatures fp32 [gamma] (device)."""
        if temps is None:
            temps = torch.empty(self.gamma, dtype=torch.float32, device=self.count.device)
        _check("dspark_sts_fit", lib().dspark_sts_fit(
            _ptr(self.s_a), _ptr(self.s_y), _ptr(self.count), self.capacity, self.gamma,
            int(iters), _ptr(temps), _ptr(self.ws), self.ws.numel(), _stream(stream)))
        return temps


class MarkovDraft:
    """Draft-side sampling of one block with a Markov head (dspark_markov_draft).
    Holds the call's workspace, zeroed once at construction; calls on one stream
    share it."""

    def __init__(self, V, device="cuda"):
        n = lib().dspark_markov_draft_workspace_size(int(V))
        if n == 0:
            raise ValueError(f"vocabulary size {V} is not supported (a multiple of 128 is needed)")
        self.V = int(V)
        self.ws = torch.zeros(n, dtype=torch.uint8, device=torch.device(device))

    def __call__(self, U, W1, W2, anchor, exp_noise, draft_tok=None, p_draft=None, stream=None):
        """U, exp_noise fp32 [B, gamma, V]; W1 bf16 [V, 256]; W2 bf16 [256, V]; anchor
        int32 [B].  Returns (draft_tok int32 [B, gamma], p_draft fp32 [B, gamma, V])."""
        B, gamma, V = U.shape
        if draft_tok is None:
            draft_tok = torch.empty(B, gamma, dtype=torch.int32, device=U.device)
        if p_draft is None:
            p_draft = torch.empty(B, gamma, V, dtype=torch.float32, device=U.device)
        _check("dspark_markov_draft", lib().dspark_markov_draft(
            _ptr(U), _ptr(W1), _ptr(W2), int(W2.shape[0]), _ptr(anchor), _ptr(exp_noise), B, gamma,
            V, _ptr(draft_tok), _ptr(p_draft), _ptr(self.ws), self.ws.numel(), _stream(stream)))
        return draft_tok, p_draft


def _host_ptr(t):
    """A pinned host tensor's address (for the mapped tier word), or None."""
    if t is None:
        return None
    if t.is_cuda or not t.is_pinned():
        raise ValueError("expected a pinned host tensor")
    return t.data_ptr()


def pack(windows, ctx_len, anchor, draft_tok, tiers, mode, cu_seqlens, M_out, tier_out, row_req,
         row_pos, row_tok, stream=None, tier_host=None):
    """``tier_host``: optional pinned host int32 tensor that also receives the tier."""
    B, gamma = draft_tok.shape
    _check("dspark_pack", lib().dspark_pack(
        _ptr(windows), _ptr(ctx_len), _ptr(anchor), _ptr(draft_tok), _ptr(tiers), tiers.numel(), B,
        gamma, int(mode), row_req.numel(), _ptr(cu_seqlens), _ptr(M_out), _ptr(tier_out),
        _host_ptr(tier_host), _ptr(row_req), _ptr(row_pos), _ptr(row_tok), _stream(stream)))


def pack_plan(windows, ctx_len, anchor, draft_tok, tiers, mode, cu_seqlens, M_out, tier_out,
              row_req, row_pos, row_tok, Hq, Hkv, d_qk, d_v, attn_max_rows, max_splits,
              attn_workspace, stream=None, max_block_rows=0, tier_host=None):
    """pack, plus the work list of the verify_attn_planned call that follows (same shape
    and workspace)."""
    B, gamma = draft_tok.shape
    _check("dspark_pack_plan", lib().dspark_pack_plan(
        _ptr(windows), _ptr(ctx_len), _ptr(anchor), _ptr(draft_tok), _ptr(tiers), tiers.numel(), B,
        gamma, int(mode), row_req.numel(), _ptr(cu_seqlens), _ptr(M_out), _ptr(tier_out),
        _host_ptr(tier_host), _ptr(row_req), _ptr(row_pos), _ptr(row_tok), int(Hq), int(Hkv),
        int(d_qk), int(d_v),
        int(attn_max_rows), int(max_splits), int(max_block_rows), _ptr(attn_workspace),
        attn_workspace.numel() * attn_workspace.element_size(), _stream(stream)))


def verify_attn_workspace_size(B, max_rows, Hq, Hkv, d_qk, d_v, max_splits,
                               max_block_rows=0) -> int:
    return lib().dspark_verify_attn_workspace_size(B, max_rows, Hq, Hkv, d_qk, d_v, max_splits,
                                                   max_block_rows)


def verify_attn(q, k_new, v_new, k_cache, v_cache, page_table, ctx_len, cu_seqlens, scale,
                max_splits, out, lse, workspace, stream=None, max_block_rows=0):
    """GQA: q [rows, Hq, 128], k/v_new [rows, Hkv, 128], caches [pages, P, Hkv, 128].
    MLA: q [rows, 128, 576], k_new [rows, 576], k_cache [pages, P, 576], v_* None."""
    _verify_attn("dspark_verify_attn", q, k_new, v_new, k_cache, v_cache, page_table, ctx_len,
                 cu_seqlens, scale, max_splits, out, lse, workspace, stream, max_block_rows)


def verify_attn_planned(q, k_new, v_new, k_cache, v_cache, page_table, ctx_len, cu_seqlens,
                        scale, max_splits, out, lse, workspace, stream=None, max_block_rows=0):
    """verify_attn over the work list that pack_plan wrote into ``workspace``."""
    _verify_attn("dspark_verify_attn_planned", q, k_new, v_new, k_cache, v_cache, page_table,
                 ctx_len, cu_seqlens, scale, max_splits, out, lse, workspace, stream,
                 max_block_rows)


def _verify_attn(name, q, k_new, v_new, k_cache, v_cache, page_table, ctx_len, cu_seqlens, scale,
                 max_splits, out, lse, workspace, stream, max_block_rows):
    max_rows, Hq, d_qk = q.shape
    mla = v_cache is None
    Hkv = 1 if mla else k_cache.shape[2]
    d_v = out.shape[2]
    B = ctx_len.numel()
    _check(name, getattr(lib(), name)(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
        _ptr(page_table), page_table.shape[1], _ptr(ctx_len), _ptr(cu_seqlens), B, max_rows, Hq,
        Hkv, d_qk, d_v, k_cache.shape[1], float(scale), int(max_splits), int(max_block_rows),
        _ptr(out), _ptr(lse),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def accept_workspace_size(B, gamma, max_rows, V) -> int:
    return lib().dspark_accept_workspace_size(B, gamma, max_rows, V)


def accept(p_target, p_draft, draft_tok, uniforms, exp_noise, windows, cu_seqlens, mode,
           accept_len, cap_len, out_tok, cstar, fallback, workspace, stream=None):
    B, gamma, V = p_draft.shape
    pdt = BF16 if p_target.dtype == torch.bfloat16 else F32
    _check("dspark_accept", lib().dspark_accept(
        _ptr(p_target), _ptr(p_draft), pdt, V, _ptr(draft_tok), _ptr(uniforms), _ptr(exp_noise),
        _ptr(windows), _ptr(cu_seqlens), int(mode), B, gamma, p_target.shape[0], _ptr(accept_len),
        _ptr(cap_len), _ptr(out_tok), _ptr(cstar), _ptr(fallback), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def accept_noalloc(p_target, p_draft, draft_tok, uniforms, exp_noise, windows, cu_seqlens, mode,
                   accept_len, cap_len, out_tok, cstar, fallback, stream=None):
    """``accept`` with the library's fixed scratch instead of a workspace argument."""
    B, gamma, V = p_draft.shape
    pdt = BF16 if p_target.dtype == torch.bfloat16 else F32
    _check("dspark_accept_noalloc", lib().dspark_accept_noalloc(
        _ptr(p_target), _ptr(p_draft), pdt, V, _ptr(draft_tok), _ptr(uniforms), _ptr(exp_noise),
        _ptr(windows), _ptr(cu_seqlens), int(mode), B, gamma, p_target.shape[0], _ptr(accept_len),
        _ptr(cap_len), _ptr(out_tok), _ptr(cstar), _ptr(fallback), _stream(stream)))


def block_accept_estimate(p_target, p_draft, draft_tok, uniforms, windows, cu_seqlens, mode,
                          accept_len, cap_len, cap_lo=None, cap_hi=None, stream=None):
    """The uncut cap's interval (cap_lo, cap_hi) int32 [B] from a step's acceptance
    outputs (dspark_block_accept_estimate)."""
    B, gamma, V = p_draft.shape
    pdt = BF16 if p_target.dtype == torch.bfloat16 else F32
    if cap_lo is None:
        cap_lo = torch.empty(B, dtype=torch.int32, device=p_draft.device)
    if cap_hi is None:
        cap_hi = torch.empty(B, dtype=torch.int32, device=p_draft.device)
    _check("dspark_block_accept_estimate", lib().dspark_block_accept_estimate(
        _ptr(p_target), _ptr(p_draft), pdt, V, _ptr(draft_tok), _ptr(uniforms), _ptr(windows),
        _ptr(cu_seqlens), _ptr(accept_len), _ptr(cap_len), int(mode), B, gamma,
        p_target.shape[0], _ptr(cap_lo), _ptr(cap_hi), _stream(stream)))
    return cap_lo, cap_hi


def compact_workspace_size(B) -> int:
    return lib().dspark_compact_workspace_size(B)


def compact(k_new, v_new, cu_seqlens, accept_len, out_tok, draft_tok, page_table, ctx_len, anchor,
            free_pages, free_top, k_cache, v_cache, committed, n_committed, workspace, stream=None):
    B, gamma = draft_tok.shape
    row_bytes = k_new[0].numel() * k_new.element_size()
    _check("dspark_compact", lib().dspark_compact(
        _ptr(k_new), _ptr(v_new), row_bytes, k_new.shape[0], _ptr(cu_seqlens), _ptr(accept_len), _ptr(out_tok),
        _ptr(draft_tok), B, gamma, k_cache.shape[1], page_table.shape[1], k_cache.shape[0],
        _ptr(page_table), _ptr(ctx_len), _ptr(anchor), _ptr(free_pages), _ptr(free_top),
        _ptr(k_cache), _ptr(v_cache), _ptr(committed), _ptr(n_committed), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


class StepDesc(ctypes.Structure):
    """dspark_step_desc (field for field)."""
    _fields_ = (
        [(n, _I) for n in ("B", "gamma", "mode", "Hq", "Hkv", "d_qk", "d_v", "page_size",
                           "max_pages", "n_pages", "V", "pdt", "max_rows", "n_tiers")]
        + [("tiers_host", _P), ("tiers", _P)]
        + [(n, _I) for n in ("conf_is_logit", "cost_len", "max_tokens", "max_splits",
                             "max_block_rows")]
        + [("scale", _F)]
        + [(n, _P) for n in ("conf", "sts_temp", "cost_table", "draft_tok", "q", "k_new", "v_new",
                             "p_target", "p_draft", "uniforms", "exp_noise", "free_pages",
                             "page_table", "ctx_len", "anchor", "free_top", "k_cache", "v_cache",
                             "windows", "a_hat", "survival", "M", "E", "cu_seqlens", "M_pack",
                             "tier",
                             "row_req", "row_pos", "row_tok", "out", "lse", "accept_len",
                             "cap_len", "out_tok", "cstar", "fallback", "committed",
                             "n_committed", "tier_host", "body_log")]
        + [("log_len", _I), ("ws_attn", _P), ("ws_attn_bytes", _Z), ("ws_accept", _P),
           ("ws_accept_bytes", _Z), ("ws_compact", _P), ("ws_compact_bytes", _Z)]
    )


class StepGraph:
    """The whole verification step as one library-built CUDA graph whose captured tier
    is chosen on the device (dspark_step_graph_*): each ``launch`` runs one step from
    the current contents of the buffers it was built on."""

    def __init__(self, desc: StepDesc, keep):
        self._keep = keep            # tensors the descriptor points into
        self._desc = desc
        h = ctypes.c_void_p()
        _check("dspark_step_graph_create",
               lib().dspark_step_graph_create(ctypes.byref(desc), ctypes.byref(h)))
        self._h = h

    def launch(self, stream=None):
        _check("dspark_step_graph_launch", lib().dspark_step_graph_launch(self._h, _stream(stream)))

    @property
    def pdl(self) -> bool:
        """True if the graph's kernels keep their programmatic dependencies."""
        return bool(lib().dspark_step_graph_flags(self._h) & 1)

    def close(self):
        if self._h:
            lib().dspark_step_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def block_rows_hint_for(gamma, Hq, Hkv, mode) -> int:
    """Rows per request the attention's query tile is sized for in ``mode`` (the
    ``max_block_rows`` hint); a request with more rows is split into row tiles (exact;
    its keys are then read once per row tile, mostly from L2).

    Static and cap-accept verify the whole block: gamma + 1.  A compact window is short
    -- a few rows -- and the smallest tile holding four block rows of G = Hq / Hkv heads
    (32 query rows: floor(32 / G) block rows for G <= 8; 64 or 128 for larger groups)
    does far less softmax work per key tile than one sized for the whole block, while
    the rare longer window takes a second row tile.  (Measured with G = 4 and 5; the
    four-row floor keeps wide groups from splitting a typical window into many row
    tiles, each of which reads the request's keys again.)"""
    G = max(1, Hq // Hkv)
    if int(mode) == COMPACT:
        for cols in (32, 64, 128):
            if cols // G >= 4:
                return min(gamma + 1, cols // G)
        return gamma + 1
    return gamma + 1


class VerifyStep:
    """Device buffers and workspaces for repeated verification steps of one shape.

    ``run`` enqueues the five calls of one step on the current stream:
    schedule -> pack (with the attention work list: pack_plan) -> verify_attn (over that
    work list: verify_attn_planned) -> accept -> compact.  The per-row inputs
    (q, k_new, v_new, p_target) are read from the packed buffers the caller
    fills; state (caches, page table, ctx_len, anchor, free stack) is updated in
    place by compact.
    """

    def __init__(self, B, gamma, Hq, Hkv, d_qk, d_v, vocab, max_rows, p_dtype=torch.float32,
                 max_splits=8, device="cuda", block_rows_hint=None):
        self.B, self.gamma, self.Hq, self.Hkv, self.d_qk, self.d_v = B, gamma, Hq, Hkv, d_qk, d_v
        self.vocab, self.max_rows, self.max_splits = vocab, max_rows, max_splits
        # the attention's query tile per mode (block_rows_hint); ``block_rows_hint``
        # fixes one hint for every mode
        if block_rows_hint is None:
            self._hints = {m: block_rows_hint_for(gamma, Hq, Hkv, m)
                           for m in (COMPACT, STATIC, CAP_ACCEPT)}
        else:
            h = int(block_rows_hint)
            self._hints = {COMPACT: h, STATIC: h, CAP_ACCEPT: h}
        self.block_rows_hint = self._hints[COMPACT]  # of the last pack call
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        self.windows = torch.zeros(B, **i32)
        self.a_hat = torch.zeros(B, gamma, dtype=torch.float32, device=dev)
        self.survival = torch.zeros(B, gamma, dtype=torch.float32, device=dev)
        self.M = torch.zeros(1, **i32)
        self.E = torch.zeros(1, dtype=torch.float64, device=dev)
        self.cu_seqlens = torch.zeros(B + 1, **i32)
        self.M_pack = torch.zeros(1, **i32)
        self.tier = torch.zeros(1, **i32)
        self.row_req = torch.zeros(max_rows, **i32)
        self.row_pos = torch.zeros(max_rows, **i32)
        self.row_tok = torch.zeros(max_rows, **i32)
        self.out = torch.zeros(max_rows, Hq, d_v, dtype=torch.float32, device=dev)
        self.lse = torch.zeros(max_rows, Hq, dtype=torch.float32, device=dev)
        self.accept_len = torch.zeros(B, **i32)
        self.cap_len = torch.zeros(B, **i32)
        self.out_tok = torch.zeros(B, **i32)
        self.fallback = torch.zeros(B, **i32)
        self.cstar = torch.zeros(B, gamma, dtype=torch.float32, device=dev)
        self.committed = torch.zeros(B, gamma + 1, **i32)
        self.n_committed = torch.zeros(B, **i32)
        # sized for the smallest tile (the most work items)
        sz = verify_attn_workspace_size(B, max_rows, Hq, Hkv, d_qk, d_v, max_splits,
                                        min(self._hints.values()))
        if sz == 0:
            raise ValueError("unsupported attention shape")
        self.ws_attn = torch.empty(sz, dtype=torch.uint8, device=dev)
        self.ws_accept = torch.empty(accept_workspace_size(B, gamma, max_rows, vocab),
                                     dtype=torch.uint8, device=dev)
        self.ws_compact = torch.empty(compact_workspace_size(B), dtype=torch.uint8, device=dev)

    def schedule(self, inp, mode, stream=None):
        schedule(inp["conf"], inp["conf_is_logit"], inp["sts_temp"], inp["cost_table"],
                 inp["max_tokens"], mode, self.windows, self.a_hat, self.M, self.E, stream,
                 survival=self.survival)

    def pack(self, inp, mode, stream=None):
        self.block_rows_hint = self.hint(mode)  # for a following attention()
        pack(self.windows, inp["ctx_len"], inp["anchor"], inp["draft_tok"], inp["tiers"], mode,
             self.cu_seqlens, self.M_pack, self.tier, self.row_req, self.row_pos, self.row_tok,
             stream)

    def attention(self, inp, stream=None):
        verify_attn(inp["q"], inp["k_new"], inp.get("v_new"), inp["k_cache"], inp.get("v_cache"),
                    inp["page_table"], inp["ctx_len"], self.cu_seqlens, inp["scale"],
                    self.max_splits, self.out, self.lse, self.ws_attn, stream,
                    max_block_rows=self.block_rows_hint)

    def hint(self, mode) -> int:
        """The block-rows hint (query tile) the step uses in ``mode``."""
        return self._hints[int(mode)]

    def pack_plan(self, inp, mode, stream=None):
        """pack, with the attention work list built in the same kernel (for attention_planned,
        which takes the query tile chosen here)."""
        self.block_rows_hint = self.hint(mode)
        pack_plan(self.windows, inp["ctx_len"], inp["anchor"], inp["draft_tok"], inp["tiers"], mode,
                  self.cu_seqlens, self.M_pack, self.tier, self.row_req, self.row_pos,
                  self.row_tok, self.Hq, self.Hkv, self.d_qk, self.d_v, self.max_rows,
                  self.max_splits, self.ws_attn, stream, max_block_rows=self.block_rows_hint)

    def attention_planned(self, inp, stream=None):
        verify_attn_planned(inp["q"], inp["k_new"], inp.get("v_new"), inp["k_cache"],
                            inp.get("v_cache"), inp["page_table"], inp["ctx_len"],
                            self.cu_seqlens, inp["scale"], self.max_splits, self.out, self.lse,
                            self.ws_attn, stream, max_block_rows=self.block_rows_hint)

    def accept(self, inp, mode, stream=None):
        accept(inp["p_target"], inp["p_draft"], inp["draft_tok"], inp["uniforms"],
               inp["exp_noise"], self.windows, self.cu_seqlens, mode, self.accept_len,
               self.cap_len, self.out_tok, self.cstar, self.fallback, self.ws_accept, stream)

    def compact(self, inp, stream=None):
        compact(inp["k_new"], inp.get("v_new"), self.cu_seqlens, self.accept_len, self.out_tok,
                inp["draft_tok"], inp["page_table"], inp["ctx_len"], inp["anchor"],
                inp["free_pages"], inp["free_top"], inp["k_cache"], inp.get("v_cache"),
                self.committed, self.n_committed, self.ws_compact, stream)

    def graph(self, inp, mode, tier_host=None, body_log=None) -> StepGraph:
        """The step on these buffers and ``inp``'s tensors as a StepGraph (tier chosen
        on the device).  ``tier_host``: optional pinned host int32 word receiving each
        step's tier; ``body_log``: optional device int32 [1 + n] recording the body
        index each launch ran (element 0 counts launches; the caller zeroes it)."""
        pdt = inp["p_target"].dtype
        tiers = inp["tiers"]
        tiers_dev = tiers.to(self.windows.device, torch.int32)
        tiers_host = tiers.cpu().to(torch.int32).contiguous()
        d = StepDesc()
        d.B, d.gamma, d.mode = self.B, self.gamma, int(mode)
        d.Hq, d.Hkv, d.d_qk, d.d_v = self.Hq, self.Hkv, self.d_qk, self.d_v
        d.page_size, d.max_pages = inp["k_cache"].shape[1], inp["page_table"].shape[1]
        d.n_pages, d.V = inp["k_cache"].shape[0], self.vocab
        d.pdt = BF16 if pdt == torch.bfloat16 else F32
        d.max_rows, d.n_tiers = self.max_rows, tiers_host.numel()
        d.tiers_host, d.tiers = tiers_host.data_ptr(), _ptr(tiers_dev)
        d.conf_is_logit, d.cost_len = int(inp["conf_is_logit"]), inp["cost_table"].numel()
        d.max_tokens, d.max_splits, d.max_block_rows = (int(inp["max_tokens"]), self.max_splits,
                                                      self.hint(mode))
        d.scale = float(inp["scale"])
        for k in ("conf", "sts_temp", "cost_table", "draft_tok", "q", "k_new", "p_target", "p_draft",
                  "uniforms", "exp_noise", "free_pages", "page_table", "ctx_len", "anchor",
                  "free_top", "k_cache"):
            setattr(d, k, _ptr(inp[k]))
        d.v_new, d.v_cache = _ptr(inp.get("v_new")), _ptr(inp.get("v_cache"))
        for k in ("windows", "a_hat", "survival", "M", "E", "cu_seqlens", "M_pack", "tier",
                  "row_req",
                  "row_pos", "row_tok", "out", "lse", "accept_len", "cap_len", "out_tok", "cstar",
                  "fallback", "committed", "n_committed"):
            setattr(d, k, _ptr(getattr(self, k)))
        d.tier_host = _host_ptr(tier_host)
        d.body_log = _ptr(body_log)
        d.log_len = 0 if body_log is None else body_log.numel() - 1
        d.ws_attn, d.ws_attn_bytes = _ptr(self.ws_attn), self.ws_attn.numel()
        d.ws_accept, d.ws_accept_bytes = _ptr(self.ws_accept), self.ws_accept.numel()
        d.ws_compact, d.ws_compact_bytes = _ptr(self.ws_compact), self.ws_compact.numel()
        return StepGraph(d, (tiers_dev, tiers_host, inp, tier_host, body_log))

    def run(self, inp, mode, stream=None):
        self.schedule(inp, mode, stream)
        self.pack_plan(inp, mode, stream)
        self.attention_planned(inp, stream)
        self.accept(inp, mode, stream)
        self.compact(inp, stream)

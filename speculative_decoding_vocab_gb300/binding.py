"""Thin Python binding of the C ABI in include/ssd.h (argument marshalling only).

Each function has the name of the C call it wraps and takes torch CUDA
tensors; it checks dtypes, derives sizes and strides, passes raw device
pointers and the current (or given) CUDA stream, and turns a non-zero status
into an exception.  Every step of the round runs in the library's kernels:
there is no fallback path, and a missing library raises at load time.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

SSD_OK, SSD_ERR_INVALID_ARG, SSD_ERR_UNSUPPORTED, SSD_ERR_WORKSPACE, SSD_ERR_CUDA = range(5)
SSD_F32, SSD_BF16 = 0, 1
FLAG_BAD_TOKEN = 1
FLAG_ZERO_RESIDUAL = 2
FLAG_WAIT_TIMEOUT = 4
FLAG_BAD_OUTCOME = 8
FLAG_BAD_TREE = 16
FLAG_BAD_BLOCK = 32
FLAG_BAD_PREFIX = 64
FLAG_BAD_HISTORY = 128
FLAG_BAD_RATE = 256

EXPORTS = ("ssd_status_string", "ssd_fanout_split", "ssd_workspace_size", "ssd_set_timing_events", "ssd_set_trace",
           "ssd_saguaro_sample",
           "ssd_verify", "ssd_verify_noalloc", "ssd_verify_noalloc_max_bytes",
           "ssd_predict_outcomes", "ssd_cache_lookup", "ssd_round", "ssd_round_analytics",
           "ssd_attention_workspace_size", "ssd_branch_attention", "ssd_ngram_backup",
           "ssd_fallback_plan", "ssd_fill_sample", "ssd_kv_append", "ssd_tree_verify",
           "ssd_round_pipelined")

_lib = None


class SSDError(RuntimeError):
    def __init__(self, call, code, msg):
        super().__init__(f"{call} failed: {msg} (status {code})")
        self.code = code


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libssd_gb300.so (built by ``build()``); raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB
    if not os.path.exists(p):
        raise RuntimeError(f"the CUDA library {p} is not built; run __graft_entry__.build() "
                           "(or python -m speculative_decoding_vocab_gb300.build) first")
    lib = ctypes.CDLL(p)
    _declare(lib)
    if path is None:
        _lib = lib
    return lib


_vp = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_f = ctypes.c_float
_d = ctypes.c_double
_sz = ctypes.c_size_t


def _declare(lib):
    lib.ssd_status_string.argtypes = [_i]
    lib.ssd_status_string.restype = ctypes.c_char_p
    lib.ssd_fanout_split.argtypes = [_i, _i, _d, _vp]
    lib.ssd_fanout_split.restype = _i
    lib.ssd_workspace_size.argtypes = [_i, _i, _i, _i, _vp]
    lib.ssd_workspace_size.restype = _sz
    lib.ssd_set_timing_events.argtypes = [_vp, _vp]
    lib.ssd_set_timing_events.restype = _i
    lib.ssd_set_trace.argtypes = [_vp, _sz]
    lib.ssd_set_trace.restype = _i
    lib.ssd_saguaro_sample.argtypes = [_vp, _i, _i64, _i64, _i, _i, _i, _vp, _f, _f, _vp, _vp, _vp,
                                       _vp, _vp, _sz, _vp]
    lib.ssd_saguaro_sample.restype = _i
    lib.ssd_verify.argtypes = [_vp, _vp, _i, _i64, _i64, _i, _i, _i, _vp, _f, _f, _vp, _vp, _vp,
                               _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
    lib.ssd_verify.restype = _i
    lib.ssd_verify_noalloc.argtypes = [_vp, _vp, _i, _i64, _i64, _i, _i, _i, _vp, _f, _f, _vp, _vp,
                                       _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.ssd_verify_noalloc.restype = _i
    lib.ssd_verify_noalloc_max_bytes.argtypes = []
    lib.ssd_verify_noalloc_max_bytes.restype = _sz
    lib.ssd_predict_outcomes.argtypes = [_vp, _i, _i64, _i64, _i, _i, _i, _vp, _f, _vp, _vp, _vp,
                                         _vp, _sz, _vp]
    lib.ssd_predict_outcomes.restype = _i
    lib.ssd_cache_lookup.argtypes = [_vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.ssd_cache_lookup.restype = _i
    lib.ssd_round.argtypes = ([_vp, _vp, _i, _i64, _i64, _i, _i, _i, _vp, _f, _f, _vp, _vp, _vp, _vp]
                              + [_vp] * 14 + [_vp, _sz, _vp])
    lib.ssd_round.restype = _i
    lib.ssd_round_pipelined.argtypes = lib.ssd_round.argtypes
    lib.ssd_round_pipelined.restype = _i
    lib.ssd_round_analytics.argtypes = ([_vp, _vp, _i, _i64, _i64, _i, _i, _i, _vp, _f, _f]
                                        + [_vp] * 7 + [_vp, _sz, _vp])
    lib.ssd_round_analytics.restype = _i
    lib.ssd_attention_workspace_size.argtypes = [_i, _i, _i, _i, _i, _i]
    lib.ssd_attention_workspace_size.restype = _sz
    lib.ssd_branch_attention.argtypes = [_vp, _vp, _vp, _vp, _i, _i64, _vp, _vp, _i, _i, _i, _i, _i,
                                         _i, _f, _vp, _vp, _vp, _vp, _sz, _vp]
    lib.ssd_branch_attention.restype = _i
    lib.ssd_fill_sample.argtypes = [_vp, _i, _i64, _i, _i, _i, _i, _f, _f, _vp, _i, _i, _vp, _vp, _vp,
                                    _vp, _vp, _sz, _vp]
    lib.ssd_fill_sample.restype = _i
    lib.ssd_kv_append.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i64, _vp, _i, _i, _i, _i, _i, _vp, _vp]
    lib.ssd_kv_append.restype = _i
    lib.ssd_tree_verify.argtypes = [_vp, _vp, _i, _i64, _i64, _i, _i, _i, _f, _vp, _vp, _vp, _vp, _vp,
                                    _vp, _vp, _vp, _vp, _vp, _vp]
    lib.ssd_tree_verify.restype = _i
    lib.ssd_ngram_backup.argtypes = [_vp, _i64, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _i, _vp, _vp,
                                     _vp, _vp]
    lib.ssd_ngram_backup.restype = _i
    lib.ssd_fallback_plan.argtypes = [_vp, _vp, _i, _d, _d, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                      _vp, _vp]
    lib.ssd_fallback_plan.restype = _i


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
def _ptr(t, dtype=None, strided=False):
    """Device address of ``t``.  The library reads every array as dense
    row-major memory of the C type its header names, so a tensor with other
    strides (unless the call passes them: ``strided``) or of another dtype is
    refused here rather than read wrongly."""
    if t is None:
        return None
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"expected a {dtype} tensor, got {t.dtype}")
    if not strided and t.numel() > 1 and not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    if not t.is_cuda:
        raise ValueError("tensors passed to the library must live on a CUDA device")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(call, code):
    if code != SSD_OK:
        msg = load().ssd_status_string(code).decode()
        raise SSDError(call, code, msg)


def _host_F(F):
    arr = (ctypes.c_int32 * len(F))(*[int(x) for x in F])
    return arr


def _logit_meta(x: torch.Tensor):
    if x.dim() != 3:
        raise ValueError("logits must be [B, K+1, V']")
    if x.numel() == 0:  # empty batch: nothing is read
        dt = SSD_F32 if x.dtype == torch.float32 else SSD_BF16
        return dt, x.shape[1] * x.shape[2], x.shape[2]
    if x.stride(2) != 1:
        raise ValueError("logits must have unit stride on the last dim")
    if x.dtype == torch.float32:
        dt = SSD_F32
    elif x.dtype == torch.bfloat16:
        dt = SSD_BF16
    else:
        raise ValueError(f"logits must be float32 or bfloat16, got {x.dtype}")
    return dt, x.stride(0), x.stride(1)


def tensor(arr, device="cuda"):
    """numpy -> torch on ``device``; uint16 arrays are taken as bf16 bit patterns."""
    import numpy as np
    arr = np.ascontiguousarray(arr)
    if arr.dtype == np.uint16:
        return torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(arr).to(device)


def pinned(arr):
    """numpy -> page-locked host tensor (uint16 arrays as bf16)."""
    import numpy as np
    arr = np.ascontiguousarray(arr)
    if arr.dtype == np.uint16:
        return torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16).pin_memory()
    return torch.from_numpy(arr).pin_memory()


def _dtype_code(dtype) -> int:
    return SSD_F32 if dtype in (torch.float32, "f32") else SSD_BF16


# ---------------------------------------------------------------------------
# the calls
# ---------------------------------------------------------------------------
def ssd_fanout_split(budget: int, K: int, r: float = 0.5):
    F = (ctypes.c_int32 * (K + 1))()
    _check("ssd_fanout_split", load().ssd_fanout_split(int(budget), int(K), float(r), F))
    return tuple(int(x) for x in F)


def ssd_set_timing_events(before=None, after=None):
    """Record torch.cuda.Event ``before``/``after`` around the statistics pass of
    every following vocabulary call (None, None clears)."""
    if before is not None and (not before.cuda_event or not after.cuda_event):
        raise ValueError("record both events once before handing them to the library "
                         "(torch creates the CUDA event lazily)")
    b = None if before is None else ctypes.c_void_p(before.cuda_event)
    a = None if after is None else ctypes.c_void_p(after.cuda_event)
    _check("ssd_set_timing_events", load().ssd_set_timing_events(b, a))


def ssd_set_trace(buf=None):
    """Record a per-entry work trace of the following vocabulary calls into the
    uint8/int64 CUDA tensor ``buf`` (None clears)."""
    if buf is None:
        _check("ssd_set_trace", load().ssd_set_trace(None, 0))
    else:
        _check("ssd_set_trace", load().ssd_set_trace(_ptr(buf), buf.numel() * buf.element_size()))


def ssd_workspace_size(B: int, K: int, V: int, dtype, F) -> int:
    return int(load().ssd_workspace_size(int(B), int(K), int(V), _dtype_code(dtype), _host_F(F)))


def workspace(B, K, V, dtype, F, device="cuda") -> torch.Tensor:
    n = ssd_workspace_size(B, K, V, dtype, F)
    if n == 0 and B > 0:
        raise SSDError("ssd_workspace_size", SSD_ERR_UNSUPPORTED, "unsupported shape")
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def ssd_saguaro_sample(draft, V, F, C, T, u_draft, d_out, qd_out=None, status=None, ws=None,
                       stream=None):
    dt, ss, rs = _logit_meta(draft)
    B, K1 = draft.shape[0], draft.shape[1]
    _check("ssd_saguaro_sample", load().ssd_saguaro_sample(
        _ptr(draft, strided=True), dt, ss, rs, B, K1 - 1, int(V), _host_F(F), float(C), float(T), _ptr(u_draft, torch.float32),
        _ptr(d_out, torch.int32), _ptr(qd_out, torch.float32), _ptr(status, torch.int32), _ptr(ws, torch.uint8), 0 if ws is None else ws.numel(),
        _stream(stream)))


def ssd_verify(target, draft, V, F, C, T, d, u_acc, u_bonus, accept_len, out_tokens, bonus,
               accept_prob=None, resid_mass=None, status=None, ws=None, stream=None, near_ties=None):
    dt, ss, rs = _logit_meta(target)
    if draft.dtype != target.dtype or draft.stride() != target.stride() or draft.shape != target.shape:
        raise ValueError("target and draft logits must share dtype, shape and strides")
    B, K1 = target.shape[0], target.shape[1]
    _check("ssd_verify", load().ssd_verify(
        _ptr(target, strided=True), _ptr(draft, strided=True), dt, ss, rs, B, K1 - 1, int(V), _host_F(F), float(C), float(T),
        _ptr(d, torch.int32), _ptr(u_acc, torch.float32), _ptr(u_bonus, torch.float32), _ptr(accept_len, torch.int32), _ptr(out_tokens, torch.int32), _ptr(bonus, torch.int32),
        _ptr(accept_prob, torch.float32), _ptr(resid_mass, torch.float32), _ptr(near_ties, torch.int32), _ptr(status, torch.int32), _ptr(ws, torch.uint8),
        0 if ws is None else ws.numel(), _stream(stream)))


def ssd_verify_noalloc(target, draft, V, F, C, T, d, u_acc, u_bonus, accept_len, out_tokens, bonus,
                       accept_prob=None, resid_mass=None, status=None, stream=None, near_ties=None):
    """ssd_verify with the library's fixed device scratch instead of a workspace
    (for callers that cannot allocate device memory)."""
    dt, ss, rs = _logit_meta(target)
    if draft.dtype != target.dtype or draft.stride() != target.stride() or draft.shape != target.shape:
        raise ValueError("target and draft logits must share dtype, shape and strides")
    B, K1 = target.shape[0], target.shape[1]
    _check("ssd_verify_noalloc", load().ssd_verify_noalloc(
        _ptr(target, strided=True), _ptr(draft, strided=True), dt, ss, rs, B, K1 - 1, int(V), _host_F(F), float(C), float(T),
        _ptr(d, torch.int32), _ptr(u_acc, torch.float32), _ptr(u_bonus, torch.float32), _ptr(accept_len, torch.int32), _ptr(out_tokens, torch.int32), _ptr(bonus, torch.int32),
        _ptr(accept_prob, torch.float32), _ptr(resid_mass, torch.float32), _ptr(near_ties, torch.int32), _ptr(status, torch.int32), _stream(stream)))


def ssd_verify_noalloc_max_bytes() -> int:
    return int(load().ssd_verify_noalloc_max_bytes())


def ssd_predict_outcomes(draft, V, F, T, guess, guess_q=None, status=None, ws=None, stream=None):
    dt, ss, rs = _logit_meta(draft)
    B, K1 = draft.shape[0], draft.shape[1]
    _check("ssd_predict_outcomes", load().ssd_predict_outcomes(
        _ptr(draft, strided=True), dt, ss, rs, B, K1 - 1, int(V), _host_F(F), float(T), _ptr(guess, torch.int32),
        _ptr(guess_q, torch.float32), _ptr(status, torch.int32), _ptr(ws, torch.uint8), 0 if ws is None else ws.numel(), _stream(stream)))


def ssd_cache_lookup(guess, payload, K, F, accept_len, bonus, slot, next_tokens=None, hits=None,
                     status=None, stream=None):
    B = guess.shape[0]
    _check("ssd_cache_lookup", load().ssd_cache_lookup(
        _ptr(guess, torch.int32), _ptr(payload, torch.int32), B, int(K), _host_F(F), _ptr(accept_len, torch.int32), _ptr(bonus, torch.int32),
        _ptr(slot, torch.int32), _ptr(next_tokens, torch.int32), _ptr(hits, torch.int32), _ptr(status, torch.int32), _stream(stream)))


def ssd_round(target, draft, V, F, C, T, u_draft, u_acc, u_bonus, d_out, accept_len, out_tokens,
              bonus, payload=None, qd_out=None, accept_prob=None, resid_mass=None, guess=None,
              guess_q=None, slot=None, next_tokens=None, hits=None, status=None, ws=None,
              stream=None, near_ties=None, pipelined=False):
    """One round (sample, verify, predict, lookup).  ``pipelined``: the call
    may overlap the previous kernels on the stream (ssd_round_pipelined; no
    buffer of this call may be in use by the previous call)."""
    dt, ss, rs = _logit_meta(target)
    if draft.dtype != target.dtype or draft.stride() != target.stride() or draft.shape != target.shape:
        raise ValueError("target and draft logits must share dtype, shape and strides")
    B, K1 = target.shape[0], target.shape[1]
    fn = load().ssd_round_pipelined if pipelined else load().ssd_round
    _check("ssd_round", fn(
        _ptr(target, strided=True), _ptr(draft, strided=True), dt, ss, rs, B, K1 - 1, int(V), _host_F(F), float(C), float(T),
        _ptr(u_draft, torch.float32), _ptr(u_acc, torch.float32), _ptr(u_bonus, torch.float32), _ptr(payload, torch.int32), _ptr(d_out, torch.int32), _ptr(qd_out, torch.float32),
        _ptr(accept_len, torch.int32), _ptr(out_tokens, torch.int32), _ptr(bonus, torch.int32), _ptr(accept_prob, torch.float32), _ptr(resid_mass, torch.float32),
        _ptr(guess, torch.int32), _ptr(guess_q, torch.float32), _ptr(slot, torch.int32), _ptr(next_tokens, torch.int32), _ptr(hits, torch.int32), _ptr(near_ties, torch.int32),
        _ptr(status, torch.int32), _ptr(ws, torch.uint8), 0 if ws is None else ws.numel(), _stream(stream)))


def ssd_round_analytics(target, draft, V, F, C, T, p_accept, hit_rate, exp_tokens, alpha=None,
                        resid_w=None, hit_mass=None, status=None, ws=None, stream=None):
    dt, ss, rs = _logit_meta(target)
    if draft.dtype != target.dtype or draft.stride() != target.stride() or draft.shape != target.shape:
        raise ValueError("target and draft logits must share dtype, shape and strides")
    B, K1 = target.shape[0], target.shape[1]
    _check("ssd_round_analytics", load().ssd_round_analytics(
        _ptr(target, strided=True), _ptr(draft, strided=True), dt, ss, rs, B, K1 - 1, int(V), _host_F(F), float(C), float(T),
        _ptr(alpha, torch.float32), _ptr(resid_w, torch.float32), _ptr(p_accept, torch.float32), _ptr(hit_mass, torch.float32), _ptr(hit_rate, torch.float32),
        _ptr(exp_tokens, torch.float32), _ptr(status, torch.int32), _ptr(ws, torch.uint8), 0 if ws is None else ws.numel(),
        _stream(stream)))


def ssd_attention_workspace_size(B, Nq, Hq, Hkv, d, max_prefix) -> int:
    return int(load().ssd_attention_workspace_size(int(B), int(Nq), int(Hq), int(Hkv), int(d),
                                                   int(max_prefix)))


def ssd_branch_attention(q, k_cache, v_cache, block_table, prefix_len, parent, out, lse=None,
                         scale=None, status=None, ws=None, stream=None):
    if q.dtype != torch.bfloat16 or k_cache.dtype != torch.bfloat16 or v_cache.dtype != torch.bfloat16:
        raise ValueError("q, k_cache and v_cache must be bfloat16")
    for t in (q, k_cache, v_cache, out):
        if not t.is_contiguous():
            raise ValueError("q, k_cache, v_cache and out must be contiguous")
    B, Nq, Hq, d = q.shape
    nb, Hkv, page, d2 = k_cache.shape
    if page != 16 or d2 != d:
        raise ValueError("k_cache must be [num_blocks, Hkv, 16, d]")
    N = parent.shape[1]
    if scale is None:
        scale = d ** -0.5
    _check("ssd_branch_attention", load().ssd_branch_attention(
        _ptr(q, torch.bfloat16), _ptr(k_cache, torch.bfloat16), _ptr(v_cache, torch.bfloat16), _ptr(block_table, torch.int32), block_table.shape[1], nb,
        _ptr(prefix_len, torch.int32), _ptr(parent, torch.int32), B, N, Nq, Hq, Hkv, d, float(scale), _ptr(out, torch.bfloat16), _ptr(lse, torch.float32),
        _ptr(status, torch.int32), _ptr(ws, torch.uint8), 0 if ws is None else ws.numel(), _stream(stream)))


def ssd_ngram_backup(hist, hist_len, n, K, V, u_rand, next_tokens, slot=None, match_pos=None,
                     plan_best=None, random_option=-1, status=None, stream=None):
    """Fill the missed rows of ``next_tokens`` [B, K] from an n-gram lookup in
    each sequence's history ``hist`` [B, cap] (int32, ``hist_len`` [B] valid),
    else random tokens floor(u_rand V)."""
    B = next_tokens.shape[0] if next_tokens is not None else u_rand.shape[0]
    stride = 0
    if hist is not None:
        if hist.dtype != torch.int32 or hist.dim() != 2 or not hist.is_contiguous():
            raise ValueError("hist must be a contiguous int32 [B, cap] tensor")
        stride = hist.shape[1]
    _check("ssd_ngram_backup", load().ssd_ngram_backup(
        _ptr(hist, torch.int32), stride, _ptr(hist_len, torch.int32), B, int(n), int(K), int(V), _ptr(slot, torch.int32), _ptr(u_rand, torch.float32),
        _ptr(plan_best, torch.int32), int(random_option), _ptr(next_tokens, torch.int32), _ptr(match_pos, torch.int32), _ptr(status, torch.int32),
        _stream(stream)))


def ssd_fallback_plan(p_hit, e_hit, T_v, T_p, T_b, e_miss, time=None, tokens=None, throughput=None,
                      speedup=None, best=None, status=None, stream=None):
    """Expected round time, tokens, throughput and speedup of each backup option
    (host lists ``T_b``, ``e_miss``) for the batch's hit probabilities ``p_hit``
    and tokens ``e_hit`` (device fp32 [B]); ``best`` gets the chosen option."""
    nopt = len(T_b)
    if len(e_miss) != nopt:
        raise ValueError("T_b and e_miss must have one entry per option")
    tb = (ctypes.c_double * max(nopt, 1))(*[float(x) for x in T_b])
    em = (ctypes.c_double * max(nopt, 1))(*[float(x) for x in e_miss])
    _check("ssd_fallback_plan", load().ssd_fallback_plan(
        _ptr(p_hit, torch.float32), _ptr(e_hit, torch.float32), p_hit.shape[0], float(T_v), float(T_p), nopt, tb, em, _ptr(time, torch.float64),
        _ptr(tokens, torch.float64), _ptr(throughput, torch.float64), _ptr(speedup, torch.float64), _ptr(best, torch.int32), _ptr(status, torch.int32), _stream(stream)))


def fill_workspace(B, S, V, dtype, F_t, device="cuda") -> torch.Tensor:
    """Workspace of one ssd_fill_sample call (B*S one-draw rows at F = F_t)."""
    return workspace(B * S, 1, V, dtype, (int(F_t), 0), device)


def ssd_fill_sample(logits, V, F_t, C, T, u, tokens, t=0, payload=None, q_out=None, status=None,
                    ws=None, stream=None):
    """Draw the next token of every branch row of ``logits`` [B, S, V'] with
    sigma_{F_t, C}; optionally write it into column ``t`` of ``payload`` [B, S, Kp]."""
    if logits.dim() != 3 or (logits.numel() and logits.stride(2) != 1):
        raise ValueError("logits must be [B, S, V'] with unit stride on the last dim")
    B, S = logits.shape[0], logits.shape[1]
    if logits.numel() and logits.stride(0) != S * logits.stride(1):
        raise ValueError("branch rows must be evenly spaced (stride(0) == S * stride(1))")
    dt = _dtype_code(logits.dtype)
    Kp = 0
    if payload is not None:
        if payload.dtype != torch.int32 or not payload.is_contiguous() or tuple(payload.shape[:2]) != (B, S):
            raise ValueError("payload must be a contiguous int32 [B, S, Kp] tensor")
        Kp = payload.shape[2]
    stride = logits.stride(1) if logits.numel() else logits.shape[2]
    _check("ssd_fill_sample", load().ssd_fill_sample(
        _ptr(logits, strided=True), dt, stride, B, S, int(V), int(F_t), float(C), float(T), _ptr(u, torch.float32), int(t), Kp,
        _ptr(tokens, torch.int32), _ptr(q_out, torch.float32), _ptr(payload, torch.int32), _ptr(status, torch.int32), _ptr(ws, torch.uint8),
        0 if ws is None else ws.numel(), _stream(stream)))


def ssd_kv_append(k_new, v_new, k_cache, v_cache, block_table, prefix_len, node0, status=None,
                  stream=None):
    """Append the rows ``k_new``/``v_new`` [B, S, Hkv, d] (bf16) at tree nodes
    node0..node0+S-1 of every sequence's paged cache."""
    for x in (k_new, v_new, k_cache, v_cache):
        if x.dtype != torch.bfloat16 or not x.is_contiguous():
            raise ValueError("k_new, v_new and the caches must be contiguous bfloat16")
    B, S, Hkv, d = k_new.shape
    _check("ssd_kv_append", load().ssd_kv_append(
        _ptr(k_new, torch.bfloat16), _ptr(v_new, torch.bfloat16), _ptr(k_cache, torch.bfloat16), _ptr(v_cache, torch.bfloat16), _ptr(block_table, torch.int32),
        block_table.shape[1], k_cache.shape[0], _ptr(prefix_len, torch.int32), int(node0), B, S, Hkv, d,
        _ptr(status, torch.int32), _stream(stream)))


def ssd_tree_verify(target, draft, V, T, parent, tokens, u_acc, u_bonus, accept_len, path, bonus,
                    out_tokens=None, resid_mass=None, status=None, stream=None):
    """Verify a token tree per sequence: logits [B, N+1, V'] (row 0 the root,
    row m+1 after node m), parent/tokens/u_acc [B, N], u_bonus [B]."""
    dt, ss, rs = _logit_meta(target)
    if draft.dtype != target.dtype or draft.stride() != target.stride() or draft.shape != target.shape:
        raise ValueError("target and draft logits must share dtype, shape and strides")
    B, N1 = target.shape[0], target.shape[1]
    _check("ssd_tree_verify", load().ssd_tree_verify(
        _ptr(target, strided=True), _ptr(draft, strided=True), dt, ss, rs, B, N1 - 1, int(V), float(T), _ptr(parent, torch.int32),
        _ptr(tokens, torch.int32), _ptr(u_acc, torch.float32), _ptr(u_bonus, torch.float32), _ptr(accept_len, torch.int32), _ptr(path, torch.int32), _ptr(bonus, torch.int32),
        _ptr(out_tokens, torch.int32), _ptr(resid_mass, torch.float32), _ptr(status, torch.int32), _stream(stream)))

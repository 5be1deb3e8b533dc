"""fp64 CPU oracle of one speculation round and of tree-masked branch attention.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline / reference leg may import this package.  The product
path (the CUDA library and its Python binding) never imports it.

The arithmetic lives in ``ssd_oracle.c`` (plain C11, double precision, no
fast-math); this module compiles it with gcc and marshals numpy arrays through
ctypes.  See the C file's header for the definitions it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libssd_oracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1
FLAG_BAD_TOKEN = 1
FLAG_ZERO_RESIDUAL = 2
FLAG_BAD_OUTCOME = 8
FLAG_BAD_TREE = 16
FLAG_BAD_BLOCK = 32
FLAG_BAD_PREFIX = 64


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libssd_oracle.so`` (gcc -O2, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = ctypes.CDLL(_LIB_PATH)
            _declare(_lib)
    return _lib


_p = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_d = ctypes.c_double


def _declare(lib):
    lib.oracle_fanout_split.argtypes = [_i, _i, _d, _p]
    lib.oracle_fanout_split.restype = _i
    lib.oracle_softmax.argtypes = [_p, _i, _d, _p]
    lib.oracle_softmax.restype = None
    lib.oracle_topf.argtypes = [_p, _i, _i, _p]
    lib.oracle_topf.restype = None
    lib.oracle_saguaro_dist.argtypes = [_p, _i, _i, _d, _d, _p, _p]
    lib.oracle_saguaro_dist.restype = None
    lib.oracle_inv_cdf.argtypes = [_p, _i, _d, _p]
    lib.oracle_inv_cdf.restype = _i
    lib.oracle_saguaro_sample.argtypes = [_p, _i, _i64, _i64, _i, _i, _i, _p, _d, _d, _p, _p, _p, _p]
    lib.oracle_saguaro_sample.restype = _i
    lib.oracle_verify.argtypes = ([_p, _p, _i, _i64, _i64, _i, _i, _i, _p, _d, _d, _p, _p, _p]
                                  + [_p] * 9)
    lib.oracle_verify.restype = _i
    lib.oracle_predict.argtypes = [_p, _i, _i64, _i64, _i, _i, _i, _p, _d, _p, _p]
    lib.oracle_predict.restype = _i
    lib.oracle_lookup.argtypes = [_p, _p, _i, _i, _p, _p, _p, _p, _p, _p]
    lib.oracle_lookup.restype = _i
    lib.oracle_round_analytics.argtypes = [_p, _p, _i, _i64, _i64, _i, _i, _i, _p, _d, _d] + [_p] * 7
    lib.oracle_round_analytics.restype = _i
    lib.oracle_branch_attention.argtypes = [_p, _p, _p, _p, _i, _i64, _p, _p, _i, _i, _i, _i, _i,
                                            _i, _d, _p, _p, _p]
    lib.oracle_branch_attention.restype = _i
    lib.oracle_ngram_backup.argtypes = [_p, _i64, _p, _i, _i, _i, _i, _p, _p, _p, _p]
    lib.oracle_ngram_backup.restype = _i
    lib.oracle_fallback_plan.argtypes = [_p, _p, _i, _d, _d, _i, _p, _p, _p, _p, _p, _p]
    lib.oracle_fallback_plan.restype = _i
    lib.oracle_kv_append.argtypes = [_p, _p, _p, _p, _p, _i, _i64, _p, _i, _i, _i, _i, _i, _p]
    lib.oracle_kv_append.restype = _i
    lib.oracle_tree_verify.argtypes = [_p, _p, _i, _i64, _i64, _i, _i, _i, _d, _p, _p, _p, _p, _p, _p,
                                       _p, _p, _p, _p, _p]
    lib.oracle_tree_verify.restype = _i


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _dtype_code(arr):
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.uint16:
        return BF16
    raise TypeError(f"logits must be float32 or uint16 (bf16 bits), got {arr.dtype}")


def _F(F):
    return _c(np.asarray(F, dtype=np.int32), np.int32)


# ---------------------------------------------------------------------------
def fanout_split(budget: int, K: int, r: float = 0.5):
    F = np.zeros(K + 1, np.int32)
    rc = _L().oracle_fanout_split(int(budget), int(K), float(r), _ptr(F))
    if rc != 0:
        raise ValueError("invalid fan-out arguments")
    return tuple(int(x) for x in F)


def softmax(z, T: float):
    z = _c(z, np.float64)
    p = np.zeros_like(z)
    _L().oracle_softmax(_ptr(z), z.size, float(T), _ptr(p))
    return p


def topf(z, F: int):
    z = _c(z, np.float64)
    out = np.zeros(F, np.int32)
    _L().oracle_topf(_ptr(z), z.size, int(F), _ptr(out))
    return out


def saguaro_dist(z, F: int, C: float, T: float):
    z = _c(z, np.float64)
    qp = np.zeros_like(z)
    ins = np.zeros(z.size, np.uint8)
    _L().oracle_saguaro_dist(_ptr(z), z.size, int(F), float(C), float(T), _ptr(qp), _ptr(ins))
    return qp, ins.astype(bool)


def inv_cdf(w, u: float):
    w = _c(w, np.float64)
    m = np.zeros(1, np.float64)
    i = _L().oracle_inv_cdf(_ptr(w), w.size, float(u), _ptr(m))
    return int(i), float(m[0])


def _strides(logits, V):
    B, K1, W = logits.shape
    return K1 * W, W


def saguaro_sample(draft, V, F, C, T, u_draft):
    """Returns (d [B,K] int32, qd [B,K] float64, margin [B,K] float64)."""
    draft = np.ascontiguousarray(draft)
    B, K1, _ = draft.shape
    K = K1 - 1
    ss, rs = _strides(draft, V)
    d = np.zeros((B, K), np.int32)
    qd = np.zeros((B, K), np.float64)
    mg = np.zeros((B, K), np.float64)
    u = _c(u_draft, np.float32)
    _L().oracle_saguaro_sample(_ptr(draft), _dtype_code(draft), ss, rs, B, K, int(V), _ptr(_F(F)),
                               float(C), float(T), _ptr(u), _ptr(d), _ptr(qd), _ptr(mg))
    return d, qd, mg


def verify(target, draft, V, F, C, T, d, u_acc, u_bonus):
    """Returns a dict of every verification output and diagnostic."""
    target = np.ascontiguousarray(target)
    draft = np.ascontiguousarray(draft)
    assert target.shape == draft.shape and target.dtype == draft.dtype
    B, K1, _ = target.shape
    K = K1 - 1
    ss, rs = _strides(target, V)
    out = dict(
        accept_len=np.zeros(B, np.int32),
        out_tokens=np.zeros((B, K + 1), np.int32),
        bonus=np.zeros(B, np.int32),
        accept_prob=np.zeros((B, K), np.float64),
        resid_mass=np.zeros(B, np.float64),
        flags=np.zeros(B, np.uint32),
        acc_margin=np.zeros((B, K), np.float64),
        bonus_margin=np.zeros(B, np.float64),
        alpha=np.zeros((B, K), np.float64),
    )
    dd = _c(d, np.int32)
    ua = _c(u_acc, np.float32)
    ub = _c(u_bonus, np.float32)
    _L().oracle_verify(_ptr(target), _ptr(draft), _dtype_code(target), ss, rs, B, K, int(V),
                       _ptr(_F(F)), float(C), float(T), _ptr(dd), _ptr(ua), _ptr(ub),
                       *[_ptr(out[k]) for k in ("accept_len", "out_tokens", "bonus", "accept_prob",
                                                "resid_mass", "flags", "acc_margin",
                                                "bonus_margin", "alpha")])
    return out


def predict(draft, V, F, T):
    draft = np.ascontiguousarray(draft)
    B, K1, _ = draft.shape
    K = K1 - 1
    ss, rs = _strides(draft, V)
    sumF = int(sum(F))
    guess = np.zeros((B, sumF), np.int32)
    gq = np.zeros((B, sumF), np.float64)
    _L().oracle_predict(_ptr(draft), _dtype_code(draft), ss, rs, B, K, int(V), _ptr(_F(F)),
                        float(T), _ptr(guess), _ptr(gq))
    return guess, gq


def lookup(guess, payload, K, F, accept_len, bonus):
    guess = _c(guess, np.int32)
    B = guess.shape[0]
    slot = np.zeros(B, np.int32)
    nxt = np.zeros((B, K), np.int32)
    flags = np.zeros(B, np.uint32)
    pl = None if payload is None else _c(payload, np.int32)
    hits = _L().oracle_lookup(_ptr(guess), _ptr(pl), B, int(K), _ptr(_F(F)),
                              _ptr(_c(accept_len, np.int32)), _ptr(_c(bonus, np.int32)),
                              _ptr(slot), _ptr(nxt), _ptr(flags))
    return dict(slot=slot, next_tokens=nxt, hits=int(hits), flags=flags)


def round_analytics(target, draft, V, F, C, T):
    """Exact analytics of the round before any draw: alpha [B,K], resid_w [B,K],
    p_accept [B,K+1] = P(a = k), hit_mass [B,K+1] = P(bonus among the depth-k
    guesses | a = k), hit_rate [B], exp_tokens [B], and hit_scale [B,K+1], the size of
    the terms whose differences make up hit_mass."""
    target = np.ascontiguousarray(target)
    draft = np.ascontiguousarray(draft)
    assert target.shape == draft.shape and target.dtype == draft.dtype
    B, K1, _ = target.shape
    K = K1 - 1
    ss, rs = _strides(target, V)
    out = dict(alpha=np.zeros((B, K)), resid_w=np.zeros((B, K)), p_accept=np.zeros((B, K + 1)),
               hit_mass=np.zeros((B, K + 1)), hit_rate=np.zeros(B), exp_tokens=np.zeros(B),
               hit_scale=np.zeros((B, K + 1)))
    _L().oracle_round_analytics(_ptr(target), _ptr(draft), _dtype_code(target), ss, rs, B, K,
                                int(V), _ptr(_F(F)), float(C), float(T),
                                *[_ptr(out[k]) for k in ("alpha", "resid_w", "p_accept", "hit_mass",
                                                         "hit_rate", "exp_tokens", "hit_scale")])
    return out


def branch_attention(q, k_cache, v_cache, block_table, prefix_len, parent, Hkv, scale=None):
    """Returns (out [B,Nq,Hq,d] float64, lse [B,Nq,Hq] float64, flags [B])."""
    q = _c(q, np.uint16)
    k_cache = _c(k_cache, np.uint16)
    v_cache = _c(v_cache, np.uint16)
    block_table = _c(block_table, np.int32)
    parent = _c(parent, np.int32)
    B, Nq, Hq, d = q.shape
    N = parent.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((B, Nq, Hq, d), np.float64)
    lse = np.zeros((B, Nq, Hq), np.float64)
    flags = np.zeros(B, np.uint32)
    _L().oracle_branch_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                 block_table.shape[1], k_cache.shape[0],
                                 _ptr(_c(prefix_len, np.int32)), _ptr(parent), B, N, Nq, Hq,
                                 int(Hkv), d, float(scale), _ptr(out), _ptr(lse), _ptr(flags))
    return out, lse, flags


def run_round(inp, T=None, C=None):
    """The whole round on the oracle: sample -> verify -> predict -> lookup."""
    spec = inp.spec
    T = spec.T if T is None else T
    C = spec.C if C is None else C
    d, qd, dm = saguaro_sample(inp.draft, spec.V, spec.F, C, T, inp.u_draft)
    v = verify(inp.target, inp.draft, spec.V, spec.F, C, T, d, inp.u_acc, inp.u_bonus)
    guess, gq = predict(inp.draft, spec.V, spec.F, T)
    lk = lookup(guess, inp.payload, spec.K, spec.F, v["accept_len"], v["bonus"])
    v.update(d=d, qd=qd, draft_margin=dm, guess=guess, guess_q=gq, slot=lk["slot"],
             next_tokens=lk["next_tokens"], hits=lk["hits"])
    return v


def ngram_backup(history, hist_len, n, K, V, slot, u_rand, next_tokens=None):
    """Backup tokens for the sequences that missed the cache (slot < 0): the
    n-gram lookup in each sequence's history, random tokens where it has no
    continuation.  Returns (next_tokens [B, K], match_pos [B]); hits keep the
    given next_tokens (zeros when none are given)."""
    history = _c(history, np.int32)
    B = history.shape[0]
    nxt = np.zeros((B, K), np.int32) if next_tokens is None else _c(next_tokens, np.int32).copy()
    mpos = np.zeros(B, np.int32)
    _L().oracle_ngram_backup(_ptr(history), history.shape[1], _ptr(_c(hist_len, np.int32)), B, int(n), int(K),
                             int(V), _ptr(_c(slot, np.int32)), _ptr(_c(u_rand, np.float32)), _ptr(nxt),
                             _ptr(mpos))
    return nxt, mpos


def fallback_plan(p_hit, e_hit, T_v, T_p, T_b, e_miss):
    """The batch speedup model per backup option: dict of time, tokens,
    throughput, speedup (arrays over the options) and best (index)."""
    p_hit = _c(p_hit, np.float32)
    e_hit = _c(e_hit, np.float32)
    T_b = _c(T_b, np.float64)
    e_miss = _c(e_miss, np.float64)
    n = len(T_b)
    out = {k: np.zeros(n) for k in ("time", "tokens", "throughput", "speedup")}
    best = _L().oracle_fallback_plan(_ptr(p_hit), _ptr(e_hit), len(p_hit), float(T_v), float(T_p), n, _ptr(T_b),
                                     _ptr(e_miss), *[_ptr(out[k]) for k in ("time", "tokens", "throughput",
                                                                            "speedup")])
    out["best"] = int(best)
    return out


def fill_sample(logits, V, F_t, C, T, u):
    """One branch-decode draw: every branch row (b, s) of ``logits`` [B, S, V']
    is sampled with the Saguaro scheme sigma_{F_t, C} (a one-row
    ``saguaro_sample``).  Returns (tokens [B, S], q' of the token, margin)."""
    logits = np.ascontiguousarray(logits)
    B, S, Vp = logits.shape
    rows = logits.reshape(B * S, 1, Vp)
    pad = np.zeros((B * S, 1, Vp), logits.dtype)
    d, qd, mg = saguaro_sample(np.concatenate([rows, pad], axis=1), V, (int(F_t), 0), C, T,
                               np.asarray(u, np.float32).reshape(B * S, 1))
    return d.reshape(B, S), qd.reshape(B, S), mg.reshape(B, S)


def kv_append(k_new, v_new, k_cache, v_cache, block_table, prefix_len, node0):
    """Append rows ``k_new``/``v_new`` [B, S, Hkv, d] (bf16 bits, uint16) to
    copies of the paged caches [num_blocks, Hkv, 16, d] at logical positions
    prefix_len[b] + node0 + i.  Returns (k_cache', v_cache', flags [B])."""
    k_new = np.ascontiguousarray(k_new, np.uint16)
    v_new = np.ascontiguousarray(v_new, np.uint16)
    kc = np.array(k_cache, np.uint16, copy=True, order="C")
    vc = np.array(v_cache, np.uint16, copy=True, order="C")
    bt = _c(block_table, np.int32)
    pl = _c(prefix_len, np.int32)
    B, S, Hkv, d = k_new.shape
    flags = np.zeros(B, np.uint32)
    _L().oracle_kv_append(_ptr(k_new), _ptr(v_new), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1],
                          kc.shape[0], _ptr(pl), int(node0), B, S, Hkv, d, _ptr(flags))
    return kc, vc, flags


def tree_verify(target, draft, V, T, parent, tokens, u_acc, u_bonus):
    """Token-tree verification; logits [B, N+1, V'] (row 0: the root, row m+1:
    after node m; a view broadcast over B with stride 0 is read as is),
    parent/tokens/u_acc [B, N], u_bonus [B].  Returns a dict of accept_len,
    path [B, N], bonus, resid_mass, flags, acc_margin [B, N], bonus_margin."""
    assert target.shape == draft.shape and target.dtype == draft.dtype
    B, N1, W = target.shape
    N = N1 - 1
    es = target.itemsize

    def base(a):
        if a.strides[0] == 0:  # one set of rows shared by every sequence
            return np.ascontiguousarray(a[0])[None], 0
        return np.ascontiguousarray(a), N1 * W
    t_arr, ss = base(target)
    d_arr, ss2 = base(draft)
    assert ss == ss2
    par = _c(parent, np.int32)
    tok = _c(tokens, np.int32)
    ua = _c(u_acc, np.float32)
    ub = _c(u_bonus, np.float32)
    out = dict(accept_len=np.zeros(B, np.int32), path=np.zeros((B, N), np.int32),
               bonus=np.zeros(B, np.int32), resid_mass=np.zeros(B, np.float64),
               flags=np.zeros(B, np.uint32), acc_margin=np.zeros((B, N), np.float64),
               bonus_margin=np.zeros(B, np.float64))
    _L().oracle_tree_verify(_ptr(t_arr), _ptr(d_arr), _dtype_code(t_arr), ss, W, B, N, int(V),
                            float(T), _ptr(par), _ptr(tok), _ptr(ua), _ptr(ub),
                            *[_ptr(out[k]) for k in ("accept_len", "path", "bonus", "resid_mass",
                                                     "flags", "acc_margin", "bonus_margin")])
    return out

"""Helpers that run the CUDA path on seeded inputs and compare it with the oracle.

Comparison rules (the tolerances a fp32 kernel can be held to against fp64):
* integer outputs (draft tokens, accept lengths, emitted and bonus tokens,
  guesses, slots, next tokens, hit counts) match exactly, except for a draw
  whose uniform lies within 1e-6 of its decision threshold in the oracle's
  exact arithmetic (|u - p/q'| for an acceptance test, the distance of u*W
  to the chosen bin's edges over W for an inverse-CDF draw); such near-ties
  are counted and the rest of that sequence is not compared;
* each stage is checked on the inputs the GPU actually produced upstream (the
  oracle verifies the GPU's draft tokens, looks up the GPU's outcomes), so one
  near-tie does not cascade;
* probabilities (q'(d), accept_prob, guess_q and the residual masses) agree
  within 1e-5 relative error;
* near-ties are counted on both sides and the counts must agree: the oracle's
  (decisions whose exact margin is below 1e-6) and the GPU's own near_ties
  output (its fp32 view of the same decisions) may differ only by decisions
  whose margin sits within rounding of the 1e-6 line: at most
  NEAR_TIE_SLACK + 5%.  Note that an inverse-CDF draw is a near-tie whenever
  its token's own probability is below 2e-6 (the window covers the whole bin),
  so on 128K-token Zipf rows several percent of the draws are near-ties; the
  differences the margins excuse are a subset of them.

The oracle runs on every host core: its C functions release the GIL, so a
thread pool over slices of the batch runs them in parallel.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
from speculative_decoding_vocab_gb300 import binding as ssd
from speculative_decoding_vocab_gb300 import workloads as w

NEAR_TIE = 1e-6
PROB_RTOL = 1e-5
NEAR_TIE_SLACK = 2

_pool = None


def oracle_pool() -> ThreadPoolExecutor:
    global _pool
    if _pool is None:
        _pool = ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1))
    return _pool


def _cat(parts):
    if isinstance(parts[0], dict):
        return {k: _cat([p[k] for p in parts]) for k in parts[0]}
    if isinstance(parts[0], tuple):
        return tuple(_cat([p[i] for p in parts]) for i in range(len(parts[0])))
    if isinstance(parts[0], np.ndarray):
        return np.concatenate(parts)
    return sum(parts)


def batched(fn, n, batch_args, *rest, **kw):
    """fn(*[a[lo:hi] for a in batch_args], *rest, **kw) over slices of the
    batch of n sequences, on every host core; results concatenated."""
    workers = oracle_pool()._max_workers
    step = max(1, -(-n // (2 * workers)))
    spans = [(lo, min(n, lo + step)) for lo in range(0, n, step)]
    if len(spans) <= 1:
        return fn(*batch_args, *rest, **kw)
    futs = [oracle_pool().submit(fn, *[a[lo:hi] for a in batch_args], *rest, **kw) for lo, hi in spans]
    return _cat([f.result() for f in futs])


def to_dev(arr, dev="cuda"):
    return ssd.tensor(arr, dev)


def prepare_round(inp: w.RoundInputs, dev="cuda", ws=None):
    """Device inputs, output buffers (filled with sentinels) and a workspace for
    one round (the fills and copies are enqueued here)."""
    spec = inp.spec
    B, K, V = spec.B, spec.K, spec.V
    sumF = int(sum(spec.F))
    i32 = dict(dtype=torch.int32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    o = dict(d=torch.full((B, K), -7, **i32), qd=torch.zeros(B, K, **f32),
             accept_len=torch.full((B,), -7, **i32), out_tokens=torch.full((B, K + 1), -7, **i32),
             bonus=torch.full((B,), -7, **i32), accept_prob=torch.zeros(B, K, **f32),
             resid_mass=torch.zeros(B, **f32), guess=torch.full((B, sumF), -7, **i32),
             guess_q=torch.zeros(B, sumF, **f32), slot=torch.full((B,), -7, **i32),
             next_tokens=torch.full((B, K), -7, **i32), hits=torch.full((1,), 12345, **i32),
             near_ties=torch.zeros(1, **i32), status=torch.zeros(1, **i32))
    if ws is None:
        ws = ssd.workspace(B, K, V, spec.dtype, spec.F, dev)
    pl = to_dev(inp.payload, dev) if inp.payload is not None else None
    o["_in"] = (to_dev(inp.target, dev), to_dev(inp.draft, dev), to_dev(inp.u_draft, dev),
                to_dev(inp.u_acc, dev), to_dev(inp.u_bonus, dev), pl, ws)
    return o


def enqueue_round(inp: w.RoundInputs, o, T=None, C=None, fused=True, pipelined=False):
    """Enqueue a prepared round (fused ssd_round -- or ssd_round_pipelined -- or
    the four separate calls) without waiting."""
    spec = inp.spec
    T = spec.T if T is None else T
    C = spec.C if C is None else C
    K, V = spec.K, spec.V
    tgt, dft, ud, ua, ub, pl, ws = o["_in"]
    if fused:
        ssd.ssd_round(tgt, dft, V, spec.F, C, T, ud, ua, ub, o["d"], o["accept_len"],
                      o["out_tokens"], o["bonus"], payload=pl, qd_out=o["qd"],
                      accept_prob=o["accept_prob"], resid_mass=o["resid_mass"], guess=o["guess"],
                      guess_q=o["guess_q"], slot=o["slot"], next_tokens=o["next_tokens"],
                      hits=o["hits"], status=o["status"], ws=ws, near_ties=o["near_ties"],
                      pipelined=pipelined)
    else:
        ssd.ssd_saguaro_sample(dft, V, spec.F, C, T, ud, o["d"], o["qd"], status=o["status"], ws=ws)
        ssd.ssd_verify(tgt, dft, V, spec.F, C, T, o["d"], ua, ub, o["accept_len"], o["out_tokens"],
                       o["bonus"], accept_prob=o["accept_prob"], resid_mass=o["resid_mass"],
                       status=o["status"], ws=ws, near_ties=o["near_ties"])
        ssd.ssd_predict_outcomes(dft, V, spec.F, T, o["guess"], o["guess_q"], status=o["status"],
                                 ws=ws)
        ssd.ssd_cache_lookup(o["guess"], pl, K, spec.F, o["accept_len"], o["bonus"], o["slot"],
                             o["next_tokens"], o["hits"], status=o["status"])
    o["_fused"] = fused
    return o


def collect_round(o):
    """The outputs of a launched round as numpy arrays (after a synchronize)."""
    res = {k: v.cpu().numpy() for k, v in o.items() if not k.startswith("_")}
    res["near_tie_scope"] = "round" if o["_fused"] else "verify"  # which decisions near_ties counts
    return res


def gpu_round(inp: w.RoundInputs, T=None, C=None, dev="cuda", fused=True, ws=None):
    """Run one round on the GPU (fused ssd_round, or the four separate calls);
    ``ws``: a workspace to use instead of a fresh one."""
    o = enqueue_round(inp, prepare_round(inp, dev, ws), T, C, fused)
    torch.cuda.synchronize()
    return collect_round(o)


def _rel_ok(a, b, rtol=PROB_RTOL, floor=1e-30):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.abs(a - b) <= rtol * np.maximum(np.abs(b), floor)


class Report:
    """near_ties: GPU / oracle differences the oracle's margins excused;
    oracle_near_ties / gpu_near_ties: the decisions each side counts as
    near-ties; decisions: the draws and acceptance tests compared."""

    def __init__(self):
        self.near_ties = 0
        self.oracle_near_ties = 0
        self.gpu_near_ties = 0
        self.decisions = 0
        self.compared = 0

    def __repr__(self):
        return (f"Report(compared={self.compared}, decisions={self.decisions}, "
                f"excused={self.near_ties}, oracle_near_ties={self.oracle_near_ties}, "
                f"gpu_near_ties={self.gpu_near_ties})")


def compare_round(inp: w.RoundInputs, g: dict, T=None, C=None, seqs=None, report=None,
                  check_lookup=True):
    """Compare GPU outputs ``g`` with the oracle on sequences ``seqs`` (all by default)."""
    spec = inp.spec
    T = spec.T if T is None else T
    C = spec.C if C is None else C
    K, V, F = spec.K, spec.V, spec.F
    rep = report or Report()
    excused0 = rep.near_ties
    idx = np.arange(spec.B) if seqs is None else np.asarray(seqs)
    if seqs is None:
        tgt, dft = inp.target, inp.draft
        ud, ua, ub = inp.u_draft, inp.u_acc, inp.u_bonus
    else:
        tgt, dft = inp.target[idx], inp.draft[idx]
        ud, ua, ub = inp.u_draft[idx], inp.u_acc[idx], inp.u_bonus[idx]
    n = len(idx)
    # --- Saguaro sampling
    od, oqd, dmar = batched(lambda d_, u_: oracle.saguaro_sample(d_, V, F, C, T, u_), n, (dft, ud))
    gd = g["d"][idx]
    skip = np.zeros(len(idx), bool)
    for i in range(len(idx)):
        for j in range(K):
            if gd[i, j] != od[i, j]:
                assert dmar[i, j] < NEAR_TIE, (
                    f"seq {idx[i]} pos {j + 1}: draft token {gd[i, j]} vs oracle {od[i, j]} "
                    f"(margin {dmar[i, j]:.3g})")
                rep.near_ties += 1
                skip[i] = True
                break
    ok = ~skip
    assert np.all(_rel_ok(g["qd"][idx][ok], oqd[ok])), "q'(d) differs beyond 1e-5 relative"
    # --- verification, on the GPU's draft tokens
    ov = batched(lambda t_, d_, g_, a_, b_: oracle.verify(t_, d_, V, F, C, T, g_, a_, b_), n,
                 (tgt, dft, gd, ua, ub))
    ga, gb = g["accept_len"][idx], g["bonus"][idx]
    for i in range(len(idx)):
        if ga[i] != ov["accept_len"][i]:
            j = min(ga[i], ov["accept_len"][i])
            assert ov["acc_margin"][i, j] < NEAR_TIE, (
                f"seq {idx[i]}: accept length {ga[i]} vs oracle {ov['accept_len'][i]} "
                f"(margin {ov['acc_margin'][i, j]:.3g})")
            rep.near_ties += 1
            skip[i] = True
            continue
        if gb[i] != ov["bonus"][i]:
            assert ov["bonus_margin"][i] < NEAR_TIE, (
                f"seq {idx[i]}: bonus {gb[i]} vs oracle {ov['bonus'][i]} "
                f"(margin {ov['bonus_margin'][i]:.3g})")
            rep.near_ties += 1
            skip[i] = True
            continue
        assert np.array_equal(g["out_tokens"][idx][i], ov["out_tokens"][i]), f"seq {idx[i]} tokens"
    assert np.all(_rel_ok(g["accept_prob"][idx], ov["accept_prob"])), "accept_prob differs"
    assert np.all(_rel_ok(g["resid_mass"][idx][~skip], ov["resid_mass"][~skip])), "resid_mass"
    # --- prediction (exact on raw logits)
    og, ogq = batched(oracle.predict, n, (dft,), V, F, T)
    assert np.array_equal(g["guess"][idx], og), "guesses differ"
    assert np.all(_rel_ok(g["guess_q"][idx], ogq)), "guess_q differs"
    # --- lookup, on the GPU's outcomes
    if check_lookup:
        ol = oracle.lookup(g["guess"][idx], None if inp.payload is None else inp.payload[idx], K, F,
                           ga, gb)
        assert np.array_equal(g["slot"][idx], ol["slot"]), "slots differ"
        assert np.array_equal(g["next_tokens"][idx], ol["next_tokens"]), "next tokens differ"
        if seqs is None:
            assert int(g["hits"][0]) == ol["hits"], "hit count differs"
    rep.compared += len(idx)
    # near-ties: the decisions actually taken whose exact margin is below 1e-6
    draws = g.get("near_tie_scope", "round") == "round"
    tests_taken = int(sum(min(int(a) + 1, K) for a in ga)) if T > 0 else 0
    o_nt = int((ov["acc_margin"] < NEAR_TIE).sum() + (ov["bonus_margin"] < NEAR_TIE).sum())
    if draws:
        o_nt += int((dmar < NEAR_TIE).sum())
    rep.decisions += (n * K if draws else 0) + tests_taken + n
    rep.oracle_near_ties += o_nt
    excused = rep.near_ties - excused0
    assert excused <= o_nt, f"{excused} differences excused but only {o_nt} near-ties"
    if "near_ties" in g and seqs is None:
        gpu_nt = int(g["near_ties"][0])
        rep.gpu_near_ties += gpu_nt
        assert abs(gpu_nt - o_nt) <= NEAR_TIE_SLACK + 0.05 * o_nt, (
            f"the GPU counted {gpu_nt} near-ties, the oracle {o_nt}")
    return rep


def gpu_attention(ai: w.AttnInputs, dev="cuda", use_ws=True, want_lse=True):
    """Run ssd_branch_attention; without a workspace the keys are not split;
    without want_lse no log-sum-exp output is passed (returned lse all NaN)."""
    q = to_dev(ai.q, dev)
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    s = ai.spec
    ws_n = ssd.ssd_attention_workspace_size(s.B, ai.Nq, s.Hq, s.Hkv, s.d, int(ai.prefix_len.max()))
    ws = torch.empty(max(ws_n, 256), dtype=torch.uint8, device=dev) if use_ws else None
    ssd.ssd_branch_attention(q, to_dev(ai.k_cache, dev), to_dev(ai.v_cache, dev),
                             to_dev(ai.block_table, dev), to_dev(ai.prefix_len, dev),
                             to_dev(ai.parent, dev), out, lse=lse if want_lse else None, status=status, ws=ws)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), int(status.item())

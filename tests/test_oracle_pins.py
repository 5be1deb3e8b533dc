"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Every check here is independent of the oracle's own code path: known-answer
vectors, hand-worked rational examples, closed forms, exhaustive enumeration,
brute force on tiny inputs, and chi-squared tests of the losslessness the pages
state (机器之心 article "全球最強推理引擎還快2倍…", section "SSD 如何實現草擬與驗證并行？":
the scheme samples exactly from the target distribution).
"""
import contextlib
import ctypes
import os
import subprocess
import tempfile
from fractions import Fraction
from itertools import product

import numpy as np
import pytest

import oracle
from speculative_decoding_vocab_gb300 import workloads as w

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------------------
# input generator pins
# ---------------------------------------------------------------------------
def test_philox_known_answers():
    for row in _golden_rows("philox4x32_10_kat.txt"):
        v = [int(x, 16) for x in row]
        out = w.philox4x32_10(np.array(v[:4], np.uint32), (v[4], v[5]))
        assert [int(x) for x in out] == v[6:10]


def test_uniforms_are_24_bit_and_in_range():
    ud, ua, ub = w.round_uniforms(0, 0, 64, 5)
    for u in (ud, ua, ub):
        assert u.dtype == np.float32
        assert np.all(u >= 0) and np.all(u < 1)
        assert np.all((u.astype(np.float64) * 2 ** 24) == np.floor(u.astype(np.float64) * 2 ** 24))
    # distinct slots draw distinct numbers
    assert not np.array_equal(ud, ua)


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(1).standard_normal(100000).astype(np.float32) * 7
    x[:4] = [1.00390625, 1.01171875, -1.00390625, 3.0]  # exact ties to even
    mine = w.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)


# ---------------------------------------------------------------------------
# fan-out split
# ---------------------------------------------------------------------------
def test_fanout_golden():
    for row in _golden_rows("fanout_split.txt"):
        budget, K, r = int(row[0]), int(row[1]), float(row[2])
        assert oracle.fanout_split(budget, K, r) == tuple(int(x) for x in row[3:])


@pytest.mark.parametrize("budget,K", [(9, 4), (32, 5), (64, 4), (16, 4), (7, 6), (1000, 3), (5, 0)])
def test_fanout_invariants(budget, K):
    F = oracle.fanout_split(budget, K, 0.5)
    assert len(F) == K + 1 and sum(F) == budget and min(F) >= 1
    assert all(F[k] >= F[k + 1] for k in range(K))  # more branches at shallow depths
    if budget >= 100 * 2 ** K:  # far from rounding, the ratio approaches 1/r
        for k in range(K):
            assert abs(F[k] / F[k + 1] - 2.0) < 0.05


def test_fanout_rejects_bad_args():
    with pytest.raises(ValueError):
        oracle.fanout_split(3, 4, 0.5)
    with pytest.raises(ValueError):
        oracle.fanout_split(9, 4, 0.0)


# ---------------------------------------------------------------------------
# softmax / top-F / sigma_{F,C} / inverse CDF
# ---------------------------------------------------------------------------
def test_softmax_two_token_closed_form():
    for T in (0.3, 1.0, 2.5):
        for a, b in ((0.0, 1.0), (3.0, -2.0), (5.5, 5.5)):
            p = oracle.softmax([a, b], T)
            assert abs(p[0] - 1.0 / (1.0 + np.exp((b - a) / T))) < 1e-15


def test_softmax_T0_is_onehot_lowest_index():
    p = oracle.softmax([1.0, 3.0, 3.0, -1.0], 0.0)
    assert list(p) == [0.0, 1.0, 0.0, 0.0]


def test_topf_bruteforce_with_ties():
    rng = np.random.default_rng(5)
    for _ in range(50):
        V = int(rng.integers(1, 40))
        z = rng.integers(-3, 4, size=V).astype(np.float64)  # many ties
        F = int(rng.integers(1, V + 1))
        ref = sorted(range(V), key=lambda i: (-z[i], i))[:F]
        assert list(oracle.topf(z, F)) == ref


def test_saguaro_worked_example():
    g = {r[0]: float(Fraction(r[1])) for r in _golden_rows("saguaro_worked_example.txt")}
    q = np.array([g["q0"], g["q1"], g["q2"]])
    qp, ins = oracle.saguaro_dist(np.log(q), 1, 0.5, 1.0)
    assert list(ins) == [True, False, False]
    assert np.allclose(qp, [g["qprime0"], g["qprime1"], g["qprime2"]], rtol=0, atol=1e-14)


def test_saguaro_invariants():
    rng = np.random.default_rng(7)
    for _ in range(40):
        V = int(rng.integers(2, 300))
        z = rng.standard_normal(V) * 2
        F = int(rng.integers(1, V + 1))
        T = float(rng.choice([0.5, 1.0, 1.7]))
        C = float(rng.choice([1.0, 0.5, 0.25, 0.01]))
        q = oracle.softmax(z, T)
        qp, ins = oracle.saguaro_dist(z, F, C, T)
        assert abs(qp.sum() - 1.0) < 1e-12
        assert ins.sum() == F
        if C == 1.0:
            assert np.array_equal(qp, q)
        # ratios: inside S scaled by C relative to outside, preserved within each side
        i_in = np.flatnonzero(ins)[0]
        out = np.flatnonzero(~ins)
        if out.size:
            k = out[0]
            assert abs((qp[i_in] / qp[k]) / (q[i_in] / q[k]) - C) < 1e-10
        # mass on S in closed form C*s / (1 - (1-C)*s)
        s = q[ins].sum()
        assert abs(qp[ins].sum() - C * s / (1 - (1 - C) * s)) < 1e-12


def test_inv_cdf_exact_frequencies():
    wts = np.array([0, 3, 0, 5, 8, 0, 16, 32], np.float64) / 64.0
    counts = np.zeros(8, int)
    n = 4096
    for k in range(n):
        i, m = oracle.inv_cdf(wts, k / n)
        c = np.cumsum(wts)
        lo = c[i - 1] if i else 0.0
        assert lo <= (k / n) * wts.sum() < c[i]
        counts[i] += 1
    assert np.array_equal(counts, (wts / wts.sum() * n).astype(int))


# ---------------------------------------------------------------------------
# near-tie margins: the oracle outputs that decide which GPU / oracle integer
# differences the parity tests excuse (the 1e-6 near-tie window), pinned to
# hand-computed values; the mutants below show that the pins have power
# ---------------------------------------------------------------------------
def _pin_inv_cdf_margin():
    """The margin is the distance of u*W to the nearer edge of the chosen bin,
    over W.  Unnormalised dyadic weights (W = 64) keep every edge and u*W exact
    in fp64, so the expected value is exact too."""
    wts = np.array([0, 3, 0, 5, 8, 0, 16, 32], np.float64)
    edges = np.concatenate([[0.0], np.cumsum(wts)])
    W = wts.sum()
    for k in range(256):
        u = k / 256
        t = u * W
        i, m = oracle.inv_cdf(wts, u)
        assert edges[i] <= t < edges[i + 1]
        expect = min(t - edges[i], edges[i + 1] - t) / W
        assert m == expect, (u, i, m, expect)


def _worked_rows():
    g = {r[0]: float(Fraction(r[1])) for r in _golden_rows("saguaro_worked_example.txt")}
    p = np.array([g["p0"], g["p1"], g["p2"]])
    q = np.array([g["q0"], g["q1"], g["q2"]])
    zt = np.stack([np.log(p), np.log(p)]).astype(np.float32)[None]
    zd = np.stack([np.log(q), np.log(q)]).astype(np.float32)[None]
    return zt, zd


def _pin_draft_margin():
    """q' = (1/3, 2/5, 4/15) (the worked sigma_{1,1/2} example, edges 0, 1/3,
    11/15, 1): u = 1/2 lands in bin 1 with distances 1/6 and 7/30; u = 1/8 in
    bin 0 (1/8, 5/24); u = 11/16 in bin 1 (17/48, 11/240).  Greedy draws have
    no margin (inf)."""
    zt, zd = _worked_rows()
    for u, expect in ((0.5, 1 / 6), (0.125, 0.125), (0.6875, 11 / 240)):
        _, _, m = oracle.saguaro_sample(zd, 3, (1, 1), 0.5, 1.0, np.array([[u]], np.float32))
        assert abs(m[0, 0] - expect) < 1e-6, (u, m[0, 0], expect)
    _, _, m = oracle.saguaro_sample(zd, 3, (1, 1), 0.5, 0.0, np.array([[0.5]], np.float32))
    assert m[0, 0] == np.inf


def _pin_verify_margins():
    """Worked example, d_1 = 1 with p/q' = 1/2: acc_margin = |u - 1/2| = 1/4
    for u = 3/4 (rejected) and u = 1/4 (accepted).  After the rejection the
    residual (0, 0, 1/3) has W = 1/3 and one bin [0, 1/3): u_bonus = 1/2 is
    1/2 of W from either edge, u_bonus = 1/8 is 1/8 from the lower one.  After
    the acceptance the bonus comes from p_2 = (1/5, 1/5, 3/5): u_bonus = 1/2
    falls in [2/5, 1), 1/10 above its lower edge."""
    zt, zd = _worked_rows()
    d = np.array([[1]], np.int32)

    def run(ua, ub, T=1.0):
        return oracle.verify(zt, zd, 3, (1, 1), 0.5, T, d, np.array([[ua]], np.float32),
                             np.array([ub], np.float32))
    rej = run(0.75, 0.5)
    assert rej["accept_len"][0] == 0
    assert abs(rej["acc_margin"][0, 0] - 0.25) < 1e-6
    assert abs(rej["bonus_margin"][0] - 0.5) < 1e-6
    assert abs(run(0.75, 0.125)["bonus_margin"][0] - 0.125) < 1e-6
    acc = run(0.25, 0.5)
    assert acc["accept_len"][0] == 1
    assert abs(acc["acc_margin"][0, 0] - 0.25) < 1e-6
    assert abs(acc["bonus_margin"][0] - 0.1) < 1e-6
    greedy = run(0.75, 0.5, T=0.0)
    assert greedy["acc_margin"][0, 0] == np.inf and greedy["bonus_margin"][0] == np.inf


def test_inv_cdf_margin_is_distance_to_nearer_edge():
    _pin_inv_cdf_margin()


def test_draft_margin_worked_example():
    _pin_draft_margin()


def test_verify_margins_worked_example():
    _pin_verify_margins()


@contextlib.contextmanager
def _mutant_oracle(old: str, new: str):
    """The oracle with one planted mistake: its C source with ``old`` replaced
    by ``new``, compiled into a temporary library that the ``oracle`` module
    uses until the block ends."""
    with open(oracle._SRC) as f:
        src = f.read()
    assert src.count(old) == 1, old
    with tempfile.TemporaryDirectory() as tmp:
        c_path = os.path.join(tmp, "mutant.c")
        so_path = os.path.join(tmp, "libmutant.so")
        with open(c_path, "w") as f:
            f.write(src.replace(old, new))
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", so_path, c_path,
                               "-lm"])
        lib = ctypes.CDLL(so_path)
        oracle._declare(lib)
        saved = oracle._L()
        oracle._lib = lib
        try:
            yield
        finally:
            oracle._lib = saved


_MARGIN_LINE = "*margin = (lo < hi ? lo : hi) / W;"


@pytest.mark.parametrize("old,new,pins", [
    (_MARGIN_LINE, "*margin = 0.0;", ("inv_cdf", "draft", "verify")),         # margin left at 0
    (_MARGIN_LINE, "*margin = (lo < hi ? hi : lo) / W;", ("inv_cdf", "draft", "verify")),  # far edge
    (_MARGIN_LINE, "*margin = (lo < hi ? lo : hi);", ("inv_cdf", "verify")),  # not divided by W
    ("fabs(u - pd / qd)", "0.0", ("verify",)),                                  # acceptance margin 0
    ("fabs(u - pd / qd)", "fabs(u - qd / pd)", ("verify",)),                    # ratio inverted
])
def test_margin_pins_catch_planted_mistakes(old, new, pins):
    run = {"inv_cdf": _pin_inv_cdf_margin, "draft": _pin_draft_margin, "verify": _pin_verify_margins}
    with _mutant_oracle(old, new):
        for name in pins:
            with pytest.raises(AssertionError):
                run[name]()
    _pin_inv_cdf_margin()  # the real oracle is back


# ---------------------------------------------------------------------------
# verification: greedy chain, worked example, residual identity
# ---------------------------------------------------------------------------
def _int_logits(rng, B, K1, V):
    return rng.integers(-4, 5, size=(B, K1, V)).astype(np.float32)


def test_greedy_chain_at_T0():
    rng = np.random.default_rng(11)
    B, K, V = 200, 5, 12
    F = (3, 2, 1, 1, 1, 1)
    zt = _int_logits(rng, B, K + 1, V)
    zd = zt.copy()
    # perturb the draft on a random subset of rows so the chain breaks at random depths
    flip = rng.random((B, K + 1)) < 0.3
    zd[flip] = _int_logits(rng, B, K + 1, V)[flip]
    ud, ua, ub = w.round_uniforms(3, 0, B, K)
    d, _, _ = oracle.saguaro_sample(zd, V, F, 0.5, 0.0, ud)
    assert np.array_equal(d, np.argmax(zd[:, :K], axis=-1))
    v = oracle.verify(zt, zd, V, F, 0.5, 0.0, d, ua, ub)
    tgt = np.argmax(zt, axis=-1)
    for b in range(B):
        a = 0
        while a < K and d[b, a] == tgt[b, a]:
            a += 1
        assert v["accept_len"][b] == a
        expect = list(d[b, :a]) + [tgt[b, a]] + [-1] * (K - a)
        assert list(v["out_tokens"][b]) == expect


def test_verify_worked_example():
    g = {r[0]: float(Fraction(r[1])) for r in _golden_rows("saguaro_worked_example.txt")}
    p = np.array([g["p0"], g["p1"], g["p2"]])
    q = np.array([g["q0"], g["q1"], g["q2"]])
    # K = 1: rows = positions 1 and 2; position 2 rows are irrelevant here
    zt = np.stack([np.log(p), np.log(p)]).astype(np.float32)[None]
    zd = np.stack([np.log(q), np.log(q)]).astype(np.float32)[None]
    # d_1 = 1: p/q' = (1/5)/(2/5) = 1/2; u = 0.75 rejects, u = 0.25 accepts
    rej = oracle.verify(zt, zd, 3, (1, 1), 0.5, 1.0, np.array([[1]]), np.array([[0.75]], np.float32),
                        np.array([0.5], np.float32))
    assert rej["accept_len"][0] == 0
    assert abs(rej["resid_mass"][0] - g["resid_mass"]) < 1e-6  # fp32-rounded logits
    assert rej["bonus"][0] == 2  # the residual's only mass
    assert abs(rej["alpha"][0, 0] - g["alpha"]) < 1e-6
    assert abs(rej["accept_prob"][0, 0] - 0.5) < 1e-6
    acc = oracle.verify(zt, zd, 3, (1, 1), 0.5, 1.0, np.array([[1]]), np.array([[0.25]], np.float32),
                        np.array([0.5], np.float32))
    assert acc["accept_len"][0] == 1 and acc["out_tokens"][0, 0] == 1


def test_residual_identity():
    """sum max(0, p - q') = sum max(0, q' - p) = 1 - alpha at the rejected row."""
    spec = w.RoundSpec(B=300, K=4, V=64, dtype="f32", recipe="gauss", T=0.8, C=0.5,
                       F=(5, 3, 2, 1, 1), target_sigma=1.5, draft_noise=1.0)
    inp = w.make_round(spec, seed=2)
    r = oracle.run_round(inp)
    seen = 0
    for b in range(spec.B):
        a = r["accept_len"][b]
        if a == spec.K:
            continue
        p = oracle.softmax(inp.target[b, a].astype(np.float64), spec.T)
        qp, _ = oracle.saguaro_dist(inp.draft[b, a].astype(np.float64), spec.F[a], spec.C, spec.T)
        W = r["resid_mass"][b]
        assert abs(W - np.maximum(qp - p, 0).sum()) < 1e-12
        assert abs(W - (1 - r["alpha"][b, a])) < 1e-12
        seen += 1
    assert seen > 50


def test_zero_residual_flag_when_p_equals_q():
    spec = w.RoundSpec(B=20, K=3, V=16, dtype="f32", recipe="gauss", T=1.0, C=1.0,
                       F=(2, 1, 1, 1), target_sigma=1.0, draft_noise=0.0)
    inp = w.make_round(spec, seed=4)
    d = np.zeros((spec.B, spec.K), np.int32)  # p == q', every test accepts since u < 1 = p/q'
    v = oracle.verify(inp.target, inp.draft, spec.V, spec.F, 1.0, 1.0, d, inp.u_acc, inp.u_bonus)
    assert np.all(v["accept_len"] == spec.K)
    # force a rejection with an invalid draft token: the residual p - p has no mass
    d[:, 1] = spec.V + 3
    v = oracle.verify(inp.target, inp.draft, spec.V, spec.F, 1.0, 1.0, d, inp.u_acc, inp.u_bonus)
    assert np.all(v["accept_len"] == 1)
    assert np.all(v["flags"] & oracle.FLAG_ZERO_RESIDUAL)
    assert np.all(v["flags"] & oracle.FLAG_BAD_TOKEN)


# ---------------------------------------------------------------------------
# losslessness (chi-squared) and exhaustive enumeration at V = 8
# ---------------------------------------------------------------------------
def _chi2_pvalue(counts, probs):
    from scipy.stats import chi2
    n = counts.sum()
    exp = probs * n
    keep = exp >= 5
    c = np.append(counts[keep], counts[~keep].sum())
    e = np.append(exp[keep], exp[~keep].sum())
    if e[-1] < 5:
        c, e = c[:-1], e[:-1]
        # fold the tiny remainder into the largest cell
        c[np.argmax(e)] += counts[~keep].sum()
        e[np.argmax(e)] += exp[~keep].sum()
    stat = ((c - e) ** 2 / e).sum()
    return chi2.sf(stat, len(c) - 1)


def _v8_rows(seed, K):
    rng = np.random.default_rng(seed)
    zt = (rng.standard_normal((K + 1, 8)) * 1.5).astype(np.float32)
    zd = (zt + rng.standard_normal((K + 1, 8)) * 0.9).astype(np.float32)
    return zt, zd


def _broadcast_round(zt, zd, n):
    return (np.broadcast_to(zt, (n,) + zt.shape).copy(), np.broadcast_to(zd, (n,) + zd.shape).copy())


P_THRESHOLD = 1e-4  # pre-registered


@pytest.mark.parametrize("C", [1.0, 0.5, 0.25])
@pytest.mark.parametrize("T", [0.6, 1.0])
def test_chi2_lossless_V8(C, T):
    K, n = 3, 200_000
    F = (3, 2, 1, 1)
    zt, zd = _v8_rows(100, K)
    tgt, dft = _broadcast_round(zt, zd, n)
    ud, ua, ub = w.round_uniforms(17, int(C * 100 + T * 10), n, K)
    d, _, _ = oracle.saguaro_sample(dft, 8, F, C, T, ud)
    v = oracle.verify(tgt, dft, 8, F, C, T, d, ua, ub)
    for j in range(K + 1):
        mask = v["accept_len"] >= j
        counts = np.bincount(v["out_tokens"][mask, j], minlength=8)
        p = oracle.softmax(zt[j].astype(np.float64), T)
        assert _chi2_pvalue(counts, p) > P_THRESHOLD, (j, counts, p * mask.sum())


def test_chi2_detects_mismatched_residual():
    """Verifying with the raw draft q (C = 1) while the draft sampled from
    sigma_{F,1/4} must break losslessness visibly: the test has power."""
    K, n = 3, 200_000
    F = (3, 2, 1, 1)
    zt, zd = _v8_rows(100, K)
    tgt, dft = _broadcast_round(zt, zd, n)
    ud, ua, ub = w.round_uniforms(17, 999, n, K)
    d, _, _ = oracle.saguaro_sample(dft, 8, F, 0.25, 1.0, ud)
    v = oracle.verify(tgt, dft, 8, F, 1.0, 1.0, d, ua, ub)
    counts = np.bincount(v["out_tokens"][:, 0], minlength=8)
    p = oracle.softmax(zt[0].astype(np.float64), 1.0)
    assert _chi2_pvalue(counts, p) < 1e-12


def _exact_outcomes(zt, zd, F, C, T):
    """P(a, b) by enumerating all V^K draft sequences (V = 8, K = 3)."""
    K = zt.shape[0] - 1
    V = zt.shape[1]
    p = [oracle.softmax(zt[j].astype(np.float64), T) for j in range(K + 1)]
    qp = [oracle.saguaro_dist(zd[j].astype(np.float64), F[j], C, T)[0] for j in range(K)]
    resid = []
    for j in range(K):
        r = np.maximum(p[j] - qp[j], 0)
        resid.append(r / r.sum())
    acc = [np.where(qp[j] > 0, np.minimum(1, p[j] / np.where(qp[j] > 0, qp[j], 1)), 1.0)
           for j in range(K)]
    Pa = np.zeros(K + 1)
    for ds in product(range(V), repeat=K):
        pr = np.prod([qp[j][ds[j]] for j in range(K)])
        run = pr
        for k in range(K):
            Pa[k] += run * (1 - acc[k][ds[k]])
            run *= acc[k][ds[k]]
        Pa[K] += run
    Pab = np.zeros((K + 1, V))
    for k in range(K):
        Pab[k] = Pa[k] * resid[k]
    Pab[K] = Pa[K] * p[K]
    alpha = [np.minimum(p[j], qp[j]).sum() for j in range(K)]
    return Pab, Pa, alpha, p


@pytest.mark.parametrize("C", [1.0, 0.5, 0.25])
def test_enumeration_V8_K3(C):
    K, n, T = 3, 200_000, 1.0
    F = (3, 2, 1, 1)
    zt, zd = _v8_rows(200, K)
    Pab, Pa, alpha, p = _exact_outcomes(zt, zd, F, C, T)
    # closed form P(a = k) = prod_{j<=k} alpha_j (1 - alpha_{k+1})
    run = 1.0
    for k in range(K + 1):
        cf = run * ((1 - alpha[k]) if k < K else 1.0)
        assert abs(Pa[k] - cf) < 1e-12
        if k < K:
            run *= alpha[k]
    # the first emitted token is exactly p_1: y_1 = d_1 when a >= 1 (probability
    # min(p, q') per token), else the residual draw
    qp1 = oracle.saguaro_dist(zd[0].astype(np.float64), F[0], C, T)[0]
    emitted1 = np.minimum(p[0], qp1) + Pab[0]
    assert np.allclose(emitted1, p[0], atol=1e-12)
    # Monte Carlo through the oracle's sample -> verify -> predict -> lookup
    tgt, dft = _broadcast_round(zt, zd, n)
    ud, ua, ub = w.round_uniforms(23, int(C * 100), n, K)
    inp = w.RoundInputs(w.RoundSpec(B=n, K=K, V=8, dtype="f32", recipe="gauss", T=T, C=C, F=F),
                        tgt, dft, ud, ua, ub, None)
    r = oracle.run_round(inp)
    cells = r["accept_len"] * 8 + r["bonus"]
    counts = np.bincount(cells, minlength=(K + 1) * 8)
    assert _chi2_pvalue(counts, Pab.reshape(-1)) > P_THRESHOLD
    # exact hit rate: the bonus lies among the F_a guesses of depth a
    guess = [oracle.topf(zd[k].astype(np.float64), F[k]) for k in range(K + 1)]
    hit = sum(Pab[a, b] for a in range(K + 1) for b in guess[a])
    mc = r["hits"] / n
    assert abs(mc - hit) < 5 * np.sqrt(hit * (1 - hit) / n)


@pytest.mark.parametrize("C,T", [(1.0, 1.0), (0.5, 1.0), (0.25, 0.6)])
def test_round_analytics_match_enumeration(C, T):
    """The analytics against the exhaustive enumeration of all 8^3 draft
    sequences at V = 8, K = 3: P(a = k), the hit rate and the expected tokens
    per round, plus alpha against the verification's own alpha."""
    K, F = 3, (3, 2, 1, 1)
    zt, zd = _v8_rows(300 + int(C * 10), K)
    Pab, Pa, alpha, p = _exact_outcomes(zt, zd, F, C, T)
    an = oracle.round_analytics(zt[None], zd[None], 8, F, C, T)
    assert np.allclose(an["p_accept"][0], Pa, rtol=0, atol=1e-12)
    assert abs(an["p_accept"][0].sum() - 1.0) < 1e-12
    assert np.allclose(an["alpha"][0], alpha, rtol=0, atol=1e-12)
    assert np.allclose(an["resid_w"][0], 1.0 - np.array(alpha), rtol=0, atol=1e-12)
    guess = [oracle.topf(zd[k].astype(np.float64), F[k]) for k in range(K + 1)]
    hit = sum(Pab[a, b] for a in range(K + 1) for b in guess[a])
    assert abs(an["hit_rate"][0] - hit) < 1e-12
    for a in range(K + 1):
        assert abs(an["hit_mass"][0, a] * Pa[a] - sum(Pab[a, b] for b in guess[a])) < 1e-12
    assert abs(an["exp_tokens"][0] - sum(Pa[k] * (k + 1) for k in range(K + 1))) < 1e-12
    qp = [oracle.saguaro_dist(zd[j].astype(np.float64), F[j], C, T)[0] for j in range(K)]
    for k in range(K):
        scale = sum(p[k + 1 - 1][b] + qp[k][b] for b in guess[k]) / (1.0 - alpha[k])
        assert abs(an["hit_scale"][0, k] - scale) < 1e-12
    ud, ua, ub = w.round_uniforms(5, 0, 1, K)
    d, _, _ = oracle.saguaro_sample(zd[None], 8, F, C, T, ud)
    v = oracle.verify(zt[None], zd[None], 8, F, C, T, d, ua, ub)
    assert np.allclose(v["alpha"][0], an["alpha"][0], rtol=0, atol=1e-14)


def test_round_analytics_greedy_and_no_drafts():
    """T = 0: alpha_j is 1 when both argmaxes agree, else 0, so the accept
    count is the greedy chain's; K = 0: the round emits one token, drawn from
    p_1, and hits when it is among the depth-0 guesses."""
    zt = np.array([[[0.0, 2.0, 1.0], [3.0, 0.0, 0.0], [0.0, 0.0, 5.0]]], np.float32)
    zd = np.array([[[0.0, 3.0, 1.0], [0.0, 4.0, 0.0], [5.0, 0.0, 0.0]]], np.float32)
    an = oracle.round_analytics(zt, zd, 3, (1, 1, 2), 0.5, 0.0)
    assert list(an["alpha"][0]) == [1.0, 0.0]
    assert list(an["p_accept"][0]) == [0.0, 1.0, 0.0]
    assert an["hit_mass"][0, 1] == 0.0 and an["hit_rate"][0] == 0.0  # argmax 0 is not draft row 2's top-1
    assert an["exp_tokens"][0] == 2.0
    z1 = np.log(np.array([[[0.5, 0.3, 0.2]]])).astype(np.float32)
    an0 = oracle.round_analytics(z1, z1, 3, (2,), 1.0, 1.0)
    assert an0["p_accept"][0, 0] == 1.0 and an0["exp_tokens"][0] == 1.0
    assert abs(an0["hit_rate"][0] - 0.8) < 1e-6


# ---------------------------------------------------------------------------
# outcome prediction and cache lookup
# ---------------------------------------------------------------------------
def test_predict_bruteforce():
    rng = np.random.default_rng(9)
    B, K, V = 6, 3, 30
    F = (5, 3, 2, 1)
    z = rng.integers(-3, 3, size=(B, K + 1, V)).astype(np.float32)
    guess, gq = oracle.predict(z, V, F, 1.0)
    for b in range(B):
        off = 0
        for k in range(K + 1):
            ref = sorted(range(V), key=lambda i: (-z[b, k, i], i))[:F[k]]
            assert list(guess[b, off:off + F[k]]) == ref
            e = np.exp(z[b, k].astype(np.float64) - z[b, k].max())
            assert np.allclose(gq[b, off:off + F[k]], e[ref] / e.sum(), rtol=1e-13)
            off += F[k]


def test_lookup_bruteforce():
    rng = np.random.default_rng(10)
    B, K, V = 500, 4, 10
    F = (4, 2, 1, 1, 1)
    sumF = sum(F)
    guess = rng.integers(0, V, size=(B, sumF)).astype(np.int32)
    payload = rng.integers(0, 1000, size=(B, sumF, K)).astype(np.int32)
    a = rng.integers(-1, K + 2, size=B).astype(np.int32)  # includes out-of-range outcomes
    bon = rng.integers(0, V, size=B).astype(np.int32)
    r = oracle.lookup(guess, payload, K, F, a, bon)
    offs = np.concatenate([[0], np.cumsum(F)])
    hits = 0
    for b in range(B):
        if a[b] < 0 or a[b] > K:
            assert r["slot"][b] == -1 and r["flags"][b] & oracle.FLAG_BAD_OUTCOME
            continue
        cand = [offs[a[b]] + i for i in range(F[a[b]]) if guess[b, offs[a[b]] + i] == bon[b]]
        s = cand[0] if cand else -1
        assert r["slot"][b] == s
        if s >= 0:
            hits += 1
            assert list(r["next_tokens"][b]) == list(payload[b, s])
        else:
            assert list(r["next_tokens"][b]) == [-1] * K
    assert r["hits"] == hits


# ---------------------------------------------------------------------------
# branch attention
# ---------------------------------------------------------------------------
def _bf(x):
    return w.bf16_bits_to_f32(x).astype(np.float64)


def _dense_reference(inp, mask_fn):
    """Dense attention over contiguous K/V gathered through the block table,
    with an explicit boolean mask from ``mask_fn(b, query_node)``."""
    s = inp.spec
    B, Nq, Hq, d = inp.q.shape
    group = Hq // s.Hkv
    out = np.zeros((B, Nq, Hq, d))
    lse = np.zeros((B, Nq, Hq))
    for b in range(B):
        L = int(inp.prefix_len[b])
        npos = L + inp.N
        blk = inp.block_table[b, np.arange(npos) // w.PAGE]
        Kc = _bf(inp.k_cache[blk, :, np.arange(npos) % w.PAGE, :])  # [npos, Hkv, d]
        Vc = _bf(inp.v_cache[blk, :, np.arange(npos) % w.PAGE, :])
        for qi in range(Nq):
            node = inp.N - Nq + qi
            mask = mask_fn(b, node)  # [npos] bool
            for h in range(Hq):
                qv = _bf(inp.q[b, qi, h])
                sc = Kc[:, h // group, :] @ qv / np.sqrt(d)
                sc = np.where(mask, sc, -np.inf)
                m = sc.max()
                e = np.exp(sc - m)
                out[b, qi, h] = e @ Vc[:, h // group, :] / e.sum()
                lse[b, qi, h] = m + np.log(e.sum())
    return out, lse


def test_attention_single_key_returns_v():
    spec = w.AttnSpec(B=2, Hq=4, Hkv=2, d=16, L=0, tree="chain", n_chain=1)
    inp = w.make_attention(spec, seed=1)
    out, lse, fl = oracle.branch_attention(inp.q, inp.k_cache, inp.v_cache, inp.block_table,
                                           inp.prefix_len, inp.parent, spec.Hkv)
    for b in range(2):
        blk = inp.block_table[b, 0]
        for h in range(4):
            assert np.array_equal(out[b, 0, h], _bf(inp.v_cache[blk, h // 2, 0]))
            qk = _bf(inp.q[b, 0, h]) @ _bf(inp.k_cache[blk, h // 2, 0])
            assert abs(lse[b, 0, h] - qk / 4.0) < 1e-12


def test_attention_equal_keys_average_visible_values():
    spec = w.AttnSpec(B=2, Hq=2, Hkv=1, d=8, L=37, tree="fanout", K=2, F=(2, 1, 1), chain_len=3)
    inp = w.make_attention(spec, seed=2)
    inp.k_cache[...] = inp.k_cache[0, 0, 0]  # every key identical -> uniform weights
    out, lse, _ = oracle.branch_attention(inp.q, inp.k_cache, inp.v_cache, inp.block_table,
                                          inp.prefix_len, inp.parent, spec.Hkv)
    parent = inp.parent[0]
    for b in range(2):
        L = int(inp.prefix_len[b])
        for qi in range(inp.Nq):
            node = inp.N - inp.Nq + qi
            vis = list(range(L))
            m = node
            path = []
            while m >= 0:
                path.append(m)
                m = parent[m]
            vis += [L + n for n in sorted(path)]
            blk = inp.block_table[b, np.array(vis) // 16]
            vals = _bf(inp.v_cache[blk, 0, np.array(vis) % 16])
            assert np.allclose(out[b, qi, 0], vals.mean(axis=0), atol=1e-12)
            sc = _bf(inp.q[b, qi, 0]) @ _bf(inp.k_cache[0, 0, 0]) / np.sqrt(8)
            assert abs(lse[b, qi, 0] - (sc + np.log(len(vis)))) < 1e-10


def test_attention_chain_is_causal():
    spec = w.AttnSpec(B=3, Hq=4, Hkv=2, d=32, L=45, tree="chain", n_chain=6, ragged_prefix=True)
    inp = w.make_attention(spec, seed=3)
    out, lse, fl = oracle.branch_attention(inp.q, inp.k_cache, inp.v_cache, inp.block_table,
                                           inp.prefix_len, inp.parent, spec.Hkv)

    def causal(b, node):
        L = int(inp.prefix_len[b])
        return np.arange(L + inp.N) <= L + node

    ref, rlse = _dense_reference(inp, causal)
    assert np.allclose(out, ref, atol=1e-12) and np.allclose(lse, rlse, atol=1e-12)
    assert not fl.any()


def test_attention_tree_matches_transitive_closure_mask():
    spec = w.AttnSpec(B=2, Hq=8, Hkv=2, d=16, L=21, tree="fanout", K=3, F=(3, 2, 1, 1),
                      chain_len=3, ragged_chains=True, ragged_prefix=True)
    inp = w.make_attention(spec, seed=4)
    out, lse, _ = oracle.branch_attention(inp.q, inp.k_cache, inp.v_cache, inp.block_table,
                                          inp.prefix_len, inp.parent, spec.Hkv)
    N = inp.N
    A = np.zeros((N, N), bool)  # A[i, j]: j is the parent of i
    for i, pi in enumerate(inp.parent[0]):
        if pi >= 0:
            A[i, pi] = True
    R = np.eye(N, dtype=bool)
    for _ in range(N):
        R = R | (R.astype(int) @ A.astype(int) > 0)

    def closure(b, node):
        L = int(inp.prefix_len[b])
        m = np.zeros(L + N, bool)
        m[:L] = True
        m[L:] = R[node]
        return m

    ref, rlse = _dense_reference(inp, closure)
    assert np.allclose(out, ref, atol=1e-12) and np.allclose(lse, rlse, atol=1e-12)


def test_attention_independent_of_block_placement():
    spec = w.AttnSpec(B=2, Hq=4, Hkv=4, d=16, L=50, tree="fanout", K=2, F=(2, 1, 1), chain_len=2)
    inp = w.make_attention(spec, seed=5)
    o1, l1, _ = oracle.branch_attention(inp.q, inp.k_cache, inp.v_cache, inp.block_table,
                                        inp.prefix_len, inp.parent, spec.Hkv)
    # move every block to a new physical slot
    nb = inp.k_cache.shape[0]
    perm = np.random.default_rng(0).permutation(nb)
    k2 = np.empty_like(inp.k_cache)
    v2 = np.empty_like(inp.v_cache)
    k2[perm] = inp.k_cache
    v2[perm] = inp.v_cache
    t2 = np.where(inp.block_table >= 0, perm[np.maximum(inp.block_table, 0)], -1).astype(np.int32)
    o2, l2, _ = oracle.branch_attention(inp.q, k2, v2, t2, inp.prefix_len, inp.parent, spec.Hkv)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_attention_flags_bad_tree_and_block():
    spec = w.AttnSpec(B=1, Hq=2, Hkv=1, d=8, L=20, tree="chain", n_chain=4)
    inp = w.make_attention(spec, seed=6)
    par = inp.parent.copy()
    par[0, 2] = 3  # a parent after the node: invalid
    _, _, fl = oracle.branch_attention(inp.q, inp.k_cache, inp.v_cache, inp.block_table,
                                       inp.prefix_len, par, spec.Hkv)
    assert fl[0] & oracle.FLAG_BAD_TREE
    tab = inp.block_table.copy()
    tab[0, 0] = 10 ** 6
    _, _, fl = oracle.branch_attention(inp.q, inp.k_cache, inp.v_cache, tab, inp.prefix_len,
                                       inp.parent, spec.Hkv)
    assert fl[0] & oracle.FLAG_BAD_BLOCK


def test_attention_prefix_past_the_table_is_hidden():
    """A prefix the block table cannot hold: positions at or past 16 * maxb are
    hidden and flagged (dense reference with those positions masked, gathered
    through a table padded with a real block); a negative prefix counts as 0."""
    spec = w.AttnSpec(B=2, Hq=4, Hkv=2, d=16, L=40, tree="chain", n_chain=4)
    inp = w.make_attention(spec, seed=8)
    maxb = inp.block_table.shape[1]
    inp.prefix_len[0] = 16 * maxb - 2  # two nodes in the table, two past it
    inp.prefix_len[1] = -5
    out, lse, fl = oracle.branch_attention(inp.q, inp.k_cache, inp.v_cache, inp.block_table,
                                           inp.prefix_len, inp.parent, spec.Hkv)
    assert fl[0] & oracle.FLAG_BAD_PREFIX and fl[1] & oracle.FLAG_BAD_PREFIX
    padded = w.AttnInputs(**{**inp.__dict__})
    padded.block_table = np.concatenate([inp.block_table, inp.block_table[:, :1]], axis=1)
    padded.prefix_len = np.maximum(inp.prefix_len, 0)

    def visible(b, node):
        L = int(padded.prefix_len[b])
        pos = np.arange(L + inp.N)
        return (pos <= L + node) & (pos < 16 * maxb)

    ref, rlse = _dense_reference(padded, visible)
    assert np.allclose(out, ref, atol=1e-12) and np.allclose(lse, rlse, atol=1e-12)


def test_oracle_is_thread_safe():
    """The parity tests run the oracle on every host core at once: threaded
    calls over slices of a batch equal one call over the whole batch."""
    from concurrent.futures import ThreadPoolExecutor
    spec = w.RoundSpec(B=48, K=3, V=3000, dtype="f32", recipe="gauss", T=1.0, C=0.5,
                       F=(40, 9, 3, 1), target_sigma=2.0, draft_noise=0.5)
    inp = w.make_round(spec, seed=12)
    whole = oracle.saguaro_sample(inp.draft, spec.V, spec.F, spec.C, spec.T, inp.u_draft)
    with ThreadPoolExecutor(max_workers=8) as ex:
        parts = list(ex.map(lambda lo: oracle.saguaro_sample(inp.draft[lo:lo + 6], spec.V, spec.F,
                                                             spec.C, spec.T, inp.u_draft[lo:lo + 6]),
                            range(0, spec.B, 6)))
    for k in range(3):
        assert np.array_equal(np.concatenate([p[k] for p in parts]), whole[k])


# ---------------------------------------------------------------------------
# miss fallback: the n-gram backup speculator and the batch speedup model
# ---------------------------------------------------------------------------
def test_ngram_backup_worked_examples():
    """Hand-worked: the suffix (1, 2, 3) last occurs earlier at position 6, so
    the proposal is h[9..12]; with n = 2 the suffix (2, 3) last occurs at 7."""
    h = np.array([[5, 1, 2, 3, 9, 9, 1, 2, 3, 7, 1, 2, 3, 0, 0]], np.int32)
    u = np.full((1, 4), 0.5, np.float32)
    nxt, m = oracle.ngram_backup(h, [13], 3, 4, 100, [-1], u)
    assert m[0] == 6 and nxt[0].tolist() == [7, 1, 2, 3]
    nxt, m = oracle.ngram_backup(h, [13], 2, 4, 100, [-1], u)
    assert m[0] == 7 and nxt[0].tolist() == [7, 1, 2, 3]
    # the continuation runs past the history: the rest comes from the random backup
    h2 = np.array([[4, 4, 8, 4, 4]], np.int32)
    nxt, m = oracle.ngram_backup(h2, [5], 2, 3, 10, [-1], np.array([[0.0, 0.25, 0.5]], np.float32))
    assert m[0] == 0 and nxt[0].tolist() == [8, 4, 4]
    nxt, m = oracle.ngram_backup(h2, [5], 2, 5, 10, [-1], np.array([[0, 0, 0, 0.25, 0.75]], np.float32))
    assert nxt[0].tolist() == [8, 4, 4, 2, 7]
    # a hit keeps its tokens; no match and too short a history are all random
    nxt, m = oracle.ngram_backup(h, [13], 3, 2, 100, [4], np.zeros((1, 2), np.float32),
                                 next_tokens=np.array([[11, 12]], np.int32))
    assert m[0] == -2 and nxt[0].tolist() == [11, 12]
    nxt, m = oracle.ngram_backup(np.array([[1, 2, 3, 4]], np.int32), [4], 2, 2, 1000, [-1],
                                 np.array([[0.5, 0.125]], np.float32))
    assert m[0] == -1 and nxt[0].tolist() == [500, 125]
    # float32(0.9) lies just below 0.9, so the exact floor of u V is 8, not 9
    nxt, m = oracle.ngram_backup(np.array([[7, 7]], np.int32), [2], 2, 1, 10, [-1], np.array([[0.9]], np.float32))
    assert m[0] == -1 and nxt[0].tolist() == [8]


def test_ngram_backup_properties_random():
    """On random histories over a small alphabet: the chosen occurrence
    matches the suffix, none after it does, and the random tokens are
    floor(u V) in exact rational arithmetic."""
    from fractions import Fraction
    rng = np.random.default_rng(7)
    B, Lmax, K, V = 64, 60, 5, 1000
    h = rng.integers(0, 4, size=(B, Lmax)).astype(np.int32)
    lens = rng.integers(0, Lmax + 1, size=B).astype(np.int32)
    slot = np.where(rng.random(B) < 0.2, 3, -1).astype(np.int32)
    u = ((rng.integers(0, 1 << 24, size=(B, K))).astype(np.float64) / (1 << 24)).astype(np.float32)
    for n in (1, 2, 3, 5):
        nxt, m = oracle.ngram_backup(h, lens, n, K, V, slot, u)
        for b in range(B):
            if slot[b] >= 0:
                assert m[b] == -2
                continue
            L = int(lens[b])
            suf = list(h[b, L - n:L]) if L >= n else None
            occ = [c for c in range(0, L - n) if suf is not None and list(h[b, c:c + n]) == suf]
            assert m[b] == (occ[-1] if occ else -1)
            for t in range(K):
                p = m[b] + n + t
                if m[b] >= 0 and p < L:
                    assert nxt[b, t] == h[b, p]
                else:
                    assert nxt[b, t] == int(Fraction(float(u[b, t])) * V)


def test_fallback_plan_closed_forms():
    """Every sequence hits: the batch never waits for a backup, so the round
    costs max(T_v, T_p) and the speedup over synchronous speculation is
    (T_p + T_v) / max(T_v, T_p).  A batch of one with a certain miss costs
    max(T_v, T_p) + T_b and yields e_miss tokens."""
    out = oracle.fallback_plan(np.ones(8), np.full(8, 3.0), 1.0, 0.4, [0.4, 0.01], [3.0, 1.0])
    assert np.allclose(out["time"], [1.0, 1.0]) and np.allclose(out["tokens"], [24.0, 24.0])
    assert np.allclose(out["speedup"], 1.4) and out["best"] == 0
    out = oracle.fallback_plan([0.0], [3.0], 1.0, 0.4, [0.4, 0.01], [2.5, 1.0])
    assert np.allclose(out["time"], [1.4, 1.01]) and np.allclose(out["tokens"], [2.5, 1.0])
    assert out["best"] == 0  # 2.5 / 1.4 > 1 / 1.01


def test_fallback_plan_matches_simulation():
    """Monte Carlo of batch rounds (independent hits; any miss stalls the batch
    on the backup) against the closed form."""
    rng = np.random.default_rng(11)
    B = 6
    p = rng.uniform(0.5, 0.99, size=B).astype(np.float32)
    eh = rng.uniform(1.5, 4.0, size=B).astype(np.float32)
    T_v, T_p, T_b, e_miss = 1.0, 0.7, [0.7, 0.02], [2.0, 1.05]
    out = oracle.fallback_plan(p, eh, T_v, T_p, T_b, e_miss)
    R = 400000
    hits = rng.random((R, B)) < p.astype(np.float64)
    anymiss = ~hits.all(axis=1)
    for o in range(2):
        t = max(T_v, T_p) + anymiss * T_b[o]
        tok = (hits * eh.astype(np.float64) + (~hits) * e_miss[o]).sum(axis=1)
        assert abs(t.mean() - out["time"][o]) < 5 * t.std() / np.sqrt(R)
        assert abs(tok.mean() - out["tokens"][o]) < 5 * tok.std() / np.sqrt(R)


def test_fallback_plan_crossover_with_batch_size():
    """With equal hit rates the chance that some sequence misses grows with the
    batch, so beyond a critical batch size the fast backup wins (and below it
    the accurate one); the winner changes exactly once."""
    T_v, T_p, T_b, e_miss = 1.0, 0.5, [0.5, 0.02], [2.8, 1.0]
    best = [oracle.fallback_plan(np.full(B, 0.9), np.full(B, 3.0), T_v, T_p, T_b, e_miss)["best"]
            for B in range(1, 200)]
    assert best[0] == 0 and best[-1] == 1
    changes = sum(1 for a, b in zip(best, best[1:]) if a != b)
    assert changes == 1


# ---------------------------------------------------------------------------
# cache fill by branch decode: the paged K/V append and the per-branch draw
# ---------------------------------------------------------------------------
def _logical(cache, block_table, b, npos):
    """Positions 0..npos-1 of sequence b gathered through the block table."""
    pos = np.arange(npos)
    return cache[block_table[b, pos // 16], :, pos % 16, :]  # [npos, Hkv, d]


def test_kv_append_matches_dense_placement():
    """Gathering the paged caches back in logical order equals a dense history
    with the new rows assigned at prefix + node0 + i (page boundaries crossed,
    pages out of order); nothing else changes."""
    rng = np.random.default_rng(3)
    B, S, Hkv, d, maxb = 3, 21, 2, 8, 6
    nb = B * maxb
    table = rng.permutation(nb).astype(np.int32).reshape(B, maxb)
    kc = rng.integers(0, 1 << 16, size=(nb, Hkv, 16, d)).astype(np.uint16)
    vc = rng.integers(0, 1 << 16, size=(nb, Hkv, 16, d)).astype(np.uint16)
    kn = rng.integers(0, 1 << 16, size=(B, S, Hkv, d)).astype(np.uint16)
    vn = rng.integers(0, 1 << 16, size=(B, S, Hkv, d)).astype(np.uint16)
    prefix = np.array([0, 13, 40], np.int32)
    node0 = 5
    k2, v2, fl = oracle.kv_append(kn, vn, kc, vc, table, prefix, node0)
    assert fl.tolist() == [0, 0, 0]
    npos = 16 * maxb
    for b in range(B):
        for new, old, got in ((kn, kc, k2), (vn, vc, v2)):
            want = _logical(old, table, b, npos).copy()
            p0 = prefix[b] + node0
            want[p0:p0 + S] = new[b]
            np.testing.assert_array_equal(_logical(got, table, b, npos), want)
    # pages outside every table stay as they were (here: none), and the touched
    # count is exactly B * S rows per head
    changed = (k2 != kc).any(axis=3).sum()
    assert changed <= B * S * Hkv


def test_kv_append_flags_and_skips():
    rng = np.random.default_rng(4)
    B, S, Hkv, d, maxb = 3, 4, 1, 4, 2
    kc = np.zeros((4, Hkv, 16, d), np.uint16)
    table = np.array([[0, 1], [2, 9], [3, 3]], np.int32)   # sequence 1: page id 9 is invalid
    kn = rng.integers(1, 1 << 16, size=(B, S, Hkv, d)).astype(np.uint16)
    prefix = np.array([30, 14, -1], np.int32)              # seq 0 runs past the table
    k2, v2, fl = oracle.kv_append(kn, kn, kc, kc, table, prefix, 0)
    assert fl.tolist() == [64, 32, 64]
    # seq 0: positions 30, 31 are written; 32, 33 are past the table
    np.testing.assert_array_equal(k2[1, 0, 14:16], kn[0, :2, 0])
    # seq 1: positions 14, 15 on page 2; 16, 17 on the invalid page: skipped
    np.testing.assert_array_equal(k2[2, 0, 14:16], kn[1, :2, 0])
    assert not k2[3].any() and not k2[0].any()


def test_fill_sample_routing():
    """Each branch row is drawn with its own uniform and the depth's F_t:
    equal logits give floor(u V) (u dyadic, so exact), and a dominant token is
    avoided only when F_t >= 1 and C is small."""
    B, S, V = 2, 5, 8
    z = np.zeros((B, S, V), np.float32)
    u = (np.arange(B * S, dtype=np.float64).reshape(B, S) % 8 + 0.5) / 8
    tok, q, _ = oracle.fill_sample(z, V, 0, 1.0, 1.0, u.astype(np.float32))
    np.testing.assert_array_equal(tok, np.floor(u * V).astype(int))
    np.testing.assert_allclose(q, 1.0 / V, rtol=1e-12)
    z2 = np.zeros((B, S, V), np.float32)
    for b in range(B):
        for s in range(S):
            z2[b, s, (3 * b + s) % V] = 6.0   # one dominant token per row
    uu = np.full((B, S), 0.3, np.float32)
    t0, q0, _ = oracle.fill_sample(z2, V, 0, 1e-4, 1.0, uu)
    t1, q1, _ = oracle.fill_sample(z2, V, 1, 1e-4, 1.0, uu)
    dom = (3 * np.arange(B)[:, None] + np.arange(S)[None, :]) % V
    assert (t0 == dom).all()          # F_t = 0: no down-weighting, the dominant token
    assert (t1 != dom).all()          # F_t = 1, C = 1e-4: the dominant token is avoided


# ---------------------------------------------------------------------------
# token-tree verification (several candidates per node)
# ---------------------------------------------------------------------------
def _tree_rows(prob_rows):
    z = np.log(np.asarray(prob_rows, np.float64)).astype(np.float32)
    return z[None]


def _pin_tree_worked_example():
    """Root: p = (1/2, 1/4, 1/4), q = (1/4, 1/2, 1/4); children 0 (token 1) and
    1.  Token 1 is tested against r = p: u q = 3/4 * 1/2 > 1/4, rejected, with
    margin |3/4 - 1/2| = 1/4; the residual is max(0, p - q) = (1/4, 0, 0), W =
    1/4, r = (1, 0, 0).  (a) child 1 = token 0: u q = 1/8 < 1, accepted
    (margin |1/2 - 4| = 7/2); node 1 is a leaf, so the bonus comes from its own
    p = (1/5, 1/5, 3/5): u = 1/2 lands in [2/5, 1) at 1/10 from the lower edge.
    (b) child 1 = token 2: r(2) = 0, rejected (margin 1/2); W = 3/4, r = (1, 0,
    0): the bonus is token 0 whatever u (margin 1/2 for u = 1/2)."""
    rows_t = [(.5, .25, .25), (.2, .2, .6), (.2, .2, .6)]
    rows_d = [(.25, .5, .25), (1 / 3, 1 / 3, 1 / 3), (1 / 3, 1 / 3, 1 / 3)]
    zt, zd = _tree_rows(rows_t), _tree_rows(rows_d)
    par = np.array([[-1, -1]], np.int32)
    ua = np.array([[0.75, 0.5]], np.float32)
    ub = np.array([0.5], np.float32)
    a = oracle.tree_verify(zt, zd, 3, 1.0, par, np.array([[1, 0]], np.int32), ua, ub)
    assert a["accept_len"][0] == 1 and a["path"][0].tolist() == [1, -1] and a["bonus"][0] == 2
    assert abs(a["acc_margin"][0, 0] - 0.25) < 1e-6 and abs(a["acc_margin"][0, 1] - 3.5) < 1e-5
    assert abs(a["bonus_margin"][0] - 0.1) < 1e-6 and a["resid_mass"][0] == 1.0
    b = oracle.tree_verify(zt, zd, 3, 1.0, par, np.array([[1, 2]], np.int32), ua, ub)
    assert b["accept_len"][0] == 0 and b["bonus"][0] == 0
    assert abs(b["acc_margin"][0, 1] - 0.5) < 1e-6
    assert abs(b["resid_mass"][0] - 0.75) < 1e-6 and abs(b["bonus_margin"][0] - 0.5) < 1e-6


def test_tree_verify_worked_example():
    _pin_tree_worked_example()


@pytest.mark.parametrize("T", [0.6, 1.0])
def test_tree_verify_chain_reduces_to_verify(T):
    """A chain tree is single-draft verification: the same accept counts and,
    away from rounding ties, the same bonus as the pinned chain verifier (C = 1)."""
    rng = np.random.default_rng(21)
    B, K, V = 300, 4, 50
    zt = (rng.standard_normal((B, K + 1, V)) * 1.5).astype(np.float32)
    zd = (zt + rng.standard_normal((B, K + 1, V)) * 0.7).astype(np.float32)
    ud, ua, ub = w.round_uniforms(5, 1, B, K)
    F = (1,) * (K + 1)
    d, _, _ = oracle.saguaro_sample(zd, V, F, 1.0, T, ud)
    v = oracle.verify(zt, zd, V, F, 1.0, T, d, ua, ub)
    par = np.broadcast_to(np.arange(-1, K - 1, dtype=np.int32), (B, K)).copy()
    t = oracle.tree_verify(zt, zd, V, T, par, d, ua, ub)
    np.testing.assert_array_equal(t["accept_len"], v["accept_len"])
    ok = t["bonus_margin"] > 1e-9
    assert ok.mean() > 0.95
    np.testing.assert_array_equal(t["bonus"][ok], v["bonus"][ok])
    for b in range(B):
        a = t["accept_len"][b]
        assert t["path"][b, :a].tolist() == list(range(a))


def test_tree_verify_greedy_walk():
    """T = 0: the walk takes the first child whose token is the target's argmax
    at the node and ends with the argmax as the bonus (brute force)."""
    rng = np.random.default_rng(8)
    B, V = 100, 6
    par1 = np.array([-1, -1, -1, 0, 0, 1, 3, 3, 6], np.int32)
    N = len(par1)
    zt = rng.integers(-3, 4, size=(B, N + 1, V)).astype(np.float32)
    zd = rng.integers(-3, 4, size=(B, N + 1, V)).astype(np.float32)
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    am = zt.argmax(axis=2)  # numpy: lowest index on ties
    for b in range(B):      # make the argmax child likely
        for m in range(N):
            if rng.random() < 0.5:
                tok[b, m] = am[b, par1[m] + 1]
    par = np.broadcast_to(par1, (B, N)).copy()
    u = rng.random((B, N)).astype(np.float32)
    t = oracle.tree_verify(zt, zd, V, 0.0, par, tok, u, rng.random(B).astype(np.float32))
    for b in range(B):
        node, walk = -1, []
        while True:
            nxt = [c for c in range(N) if par1[c] == node and tok[b, c] == am[b, node + 1]]
            if not nxt:
                break
            node = nxt[0]
            walk.append(node)
        assert t["path"][b, :len(walk)].tolist() == walk and t["accept_len"][b] == len(walk)
        assert t["bonus"][b] == am[b, node + 1]


_TREE_PAR = np.array([-1, -1, -1, 0, 0, 1, 1, 2, 2], np.int32)  # 3 children, 2 each


def _tree_chi2_counts(T, n=200_000, seed=31):
    """First emitted token over n independent walks of one tree whose children
    are drawn i.i.d. from the draft at their parent."""
    rng = np.random.default_rng(seed)
    V, N = 6, len(_TREE_PAR)
    zt = (rng.standard_normal((N + 1, V)) * 1.2).astype(np.float32)
    zd = (zt + rng.standard_normal((N + 1, V)) * 1.0).astype(np.float32)
    q = [oracle.softmax(zd[r].astype(np.float64), T) for r in range(N + 1)]
    tok = np.zeros((n, N), np.int32)
    for m in range(N):
        cdf = np.cumsum(q[_TREE_PAR[m] + 1])
        tok[:, m] = np.minimum(np.searchsorted(cdf, rng.random(n) * cdf[-1], side="right"), V - 1)
    par = np.broadcast_to(_TREE_PAR, (n, N))
    t = oracle.tree_verify(np.broadcast_to(zt, (n, N + 1, V)), np.broadcast_to(zd, (n, N + 1, V)),
                           V, T, par, tok, rng.random((n, N)).astype(np.float32),
                           rng.random(n).astype(np.float32))
    first = np.where(t["accept_len"] > 0, tok[np.arange(n), np.maximum(t["path"][:, 0], 0)],
                     t["bonus"])
    return np.bincount(first, minlength=V), oracle.softmax(zt[0].astype(np.float64), T)


@pytest.mark.parametrize("T", [0.6, 1.0])
def test_tree_verify_chi2_lossless(T):
    counts, p = _tree_chi2_counts(T)
    assert _chi2_pvalue(counts, p) > P_THRESHOLD


def test_tree_verify_chi2_detects_stale_residual():
    """Testing every sibling against p (no residual update) over-emits the
    draft's favourites: the chi-squared test has power."""
    with _mutant_oracle("for (int i = 0; i < V; i++) r[i] = (r[i] > q[i]) ? (r[i] - q[i]) / W : 0.0;",
                        "(void)W;"):
        counts, p = _tree_chi2_counts(1.0)
    assert _chi2_pvalue(counts, p) < 1e-12


def test_tree_verify_flags():
    zt = np.zeros((1, 4, 5), np.float32)
    par = np.array([[-1, 5, 0]], np.int32)        # node 1's parent is past it
    tok = np.array([[9, 1, 2]], np.int32)         # node 0's token is outside [0, 5)
    t = oracle.tree_verify(zt, zt, 5, 1.0, par, tok, np.zeros((1, 3), np.float32),
                           np.zeros(1, np.float32))
    assert t["flags"][0] == 16 | 1
    assert t["accept_len"][0] == 0

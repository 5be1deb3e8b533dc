"""GPU parity of the speculation-cache fill by branch decode against the
oracle: the per-branch Saguaro draw (ssd_fill_sample: tokens bit-exact
outside near-ties, q' within 1e-5 relative, payload columns), the paged K/V
append (ssd_kv_append: caches bit-exact, flags) and the whole step loop
(append -> tree attention -> draw) over K steps."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_vocab_gb300 import binding as ssd
from speculative_decoding_vocab_gb300 import workloads as w

from parity import NEAR_TIE, PROB_RTOL, batched, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_vocab_gb300 import build
    build.build()
    ssd.load()


def gpu_fill_sample(spec, logits, t, u, payload=None):
    B, S = spec.B, spec.S
    lg = to_dev(logits)
    tok = torch.full((B, S), -7, dtype=torch.int32, device="cuda")
    q = torch.full((B, S), -1.0, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = ssd.fill_workspace(B, S, spec.V, spec.dtype, spec.F[t])
    ssd.ssd_fill_sample(lg, spec.V, spec.F[t], spec.C, spec.T, to_dev(u), tok, t=t, payload=payload,
                        q_out=q, status=st, ws=ws)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), q.cpu().numpy().astype(np.float64), int(st.item())


def check_draws(spec, logits, t, u, tok, q):
    ref_t, ref_q, mg = batched(lambda lg, uu: oracle.fill_sample(lg, spec.V, spec.F[t], spec.C,
                                                                 spec.T, uu), spec.B, (logits, u))
    ok = mg >= NEAR_TIE
    assert ok.mean() > 0.8  # Zipf rows: draws of tokens below 2e-6 are near-ties by definition
    np.testing.assert_array_equal(tok[ok], ref_t[ok])
    np.testing.assert_allclose(q[ok], ref_q[ok], rtol=PROB_RTOL, atol=0)
    return int((~ok).sum())


@pytest.mark.parametrize("t", [0, 1, 3])
def test_fill_sample_tiny(t):
    spec = w.tiny_fill()
    logits = w.fill_step_logits(spec, 5, t)
    u = w.fill_uniforms(5, 0, t, spec.B, spec.S)
    payload = torch.full((spec.B, spec.S, spec.K), -3, dtype=torch.int32, device="cuda")
    tok, q, st = gpu_fill_sample(spec, logits, t, u, payload)
    assert st == 0
    check_draws(spec, logits, t, u, tok, q)
    pl = payload.cpu().numpy()
    np.testing.assert_array_equal(pl[:, :, t], tok)
    assert (np.delete(pl, t, axis=2) == -3).all()


@pytest.mark.parametrize("T,C", [(1.0, 1.0), (0.0, 0.5), (0.6, 0.25)])
def test_fill_sample_tiny_T_C(T, C):
    import dataclasses
    spec = dataclasses.replace(w.tiny_fill(), T=T, C=C)
    logits = w.fill_step_logits(spec, 6, 0)
    u = w.fill_uniforms(6, 0, 0, spec.B, spec.S)
    tok, q, st = gpu_fill_sample(spec, logits, 0, u)
    assert st == 0
    check_draws(spec, logits, 0, u, tok, q)


def test_fill_sample_llama3_full_batch():
    """One decode step of the Llama-3 fill at full size (256 branch rows of
    128256 bf16 logits, F_1 = 4): every row against the oracle."""
    spec = w.llama3_fill()
    t = 1
    logits = w.fill_step_logits(spec, 9, t)
    u = w.fill_uniforms(9, 0, t, spec.B, spec.S)
    tok, q, st = gpu_fill_sample(spec, logits, t, u)
    assert st == 0
    check_draws(spec, logits, t, u, tok, q)


def test_fill_sample_argument_checks():
    spec = w.tiny_fill()
    lg = torch.zeros(spec.B, spec.S, spec.V, device="cuda")
    u = torch.zeros(spec.B, spec.S, device="cuda")
    tok = torch.zeros(spec.B, spec.S, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = ssd.fill_workspace(spec.B, spec.S, spec.V, "f32", 2)
    with pytest.raises(ssd.SSDError):  # C outside (0, 1]
        ssd.ssd_fill_sample(lg, spec.V, 2, 0.0, 1.0, u, tok, status=st, ws=ws)
    with pytest.raises(ssd.SSDError):  # column past the payload
        pl = torch.zeros(spec.B, spec.S, 2, dtype=torch.int32, device="cuda")
        ssd.ssd_fill_sample(lg, spec.V, 2, 0.5, 1.0, u, tok, t=2, payload=pl, status=st, ws=ws)
    with pytest.raises(ssd.SSDError):  # workspace too small
        ssd.ssd_fill_sample(lg, spec.V, 2, 0.5, 1.0, u, tok, status=st, ws=ws[:64])
    # empty batch: nothing runs
    ssd.ssd_fill_sample(lg[:0], spec.V, 2, 0.5, 1.0, u[:0], tok[:0], status=st, ws=ws)


# ---------------------------------------------------------------------------
# the paged K/V append
# ---------------------------------------------------------------------------
def bf16_normal(rng, shape):
    return w.f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32))


def caches(rng, nb, Hkv, d):
    return bf16_normal(rng, (nb, Hkv, 16, d)), bf16_normal(rng, (nb, Hkv, 16, d))


@pytest.mark.parametrize("d", [64, 128, 8])
def test_kv_append(d):
    rng = np.random.default_rng(d)
    B, S, Hkv, maxb = 5, 23, 3, 7
    nb = B * maxb + 3
    table = rng.permutation(nb)[:B * maxb].astype(np.int32).reshape(B, maxb)
    kc, vc = caches(rng, nb, Hkv, d)
    kn, vn = bf16_normal(rng, (B, S, Hkv, d)), bf16_normal(rng, (B, S, Hkv, d))
    prefix = np.array([0, 5, 16, 31, 60], np.int32)
    node0 = 9
    gk, gv = to_dev(kc), to_dev(vc)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ssd.ssd_kv_append(to_dev(kn), to_dev(vn), gk, gv, to_dev(table), to_dev(prefix), node0, status=st)
    torch.cuda.synchronize()
    rk, rv, fl = oracle.kv_append(kn, vn, kc, vc, table, prefix, node0)
    assert int(st.item()) == 0 and fl.tolist() == [0] * B
    np.testing.assert_array_equal(gk.cpu().view(torch.int16).numpy().view(np.uint16), rk)
    np.testing.assert_array_equal(gv.cpu().view(torch.int16).numpy().view(np.uint16), rv)


def test_kv_append_flags():
    rng = np.random.default_rng(2)
    B, S, Hkv, d, maxb = 3, 6, 2, 64, 2
    kc, vc = caches(rng, 4, Hkv, d)
    table = np.array([[0, 1], [2, 9], [3, 3]], np.int32)
    kn, vn = bf16_normal(rng, (B, S, Hkv, d)), bf16_normal(rng, (B, S, Hkv, d))
    prefix = np.array([28, 12, -2], np.int32)
    gk, gv = to_dev(kc), to_dev(vc)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ssd.ssd_kv_append(to_dev(kn), to_dev(vn), gk, gv, to_dev(table), to_dev(prefix), 0, status=st)
    torch.cuda.synchronize()
    rk, rv, fl = oracle.kv_append(kn, vn, kc, vc, table, prefix, 0)
    assert int(st.item()) == (ssd.FLAG_BAD_PREFIX | ssd.FLAG_BAD_BLOCK)
    assert fl.tolist() == [64, 32, 64]
    np.testing.assert_array_equal(gk.cpu().view(torch.int16).numpy().view(np.uint16), rk)
    np.testing.assert_array_equal(gv.cpu().view(torch.int16).numpy().view(np.uint16), rv)


# ---------------------------------------------------------------------------
# the step loop
# ---------------------------------------------------------------------------
def test_fill_step_loop_tiny():
    """K decode steps: append the fed nodes, tree attention with the fed nodes
    as queries, draw the next tokens into the payload.  Caches, attention
    outputs and payload against the oracle at every step."""
    spec = w.tiny_fill()
    B, K, S, Hq, Hkv, d = spec.B, spec.K, spec.S, spec.Hq, spec.Hkv, spec.d
    rng = np.random.default_rng(17)
    Nmax = K + K * S
    maxb = (spec.L + Nmax + 15) // 16
    nb = B * maxb
    table = rng.permutation(nb).astype(np.int32).reshape(B, maxb)
    prefix = np.array([spec.L, spec.L - 11], np.int32)
    kc, vc = caches(rng, nb, Hkv, d)
    gk, gv = to_dev(kc), to_dev(vc)
    gtable, gprefix = to_dev(table), to_dev(prefix)
    payload = torch.full((B, S, K), -3, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = None
    ref_payload = np.full((B, S, K), -3, np.int32)
    for t in range(K):
        kn, vn = w.fill_step_kv(spec, 3, t)
        node0 = K + t * S
        ssd.ssd_kv_append(to_dev(kn), to_dev(vn), gk, gv, gtable, gprefix, node0, status=st)
        kc, vc, fl = oracle.kv_append(kn, vn, kc, vc, table, prefix, node0)
        assert fl.tolist() == [0] * B
        parent = np.broadcast_to(w.fill_tree(K, spec.F, t + 1), (B, node0 + S)).copy()
        q = w.f32_to_bf16_bits(rng.standard_normal((B, S, Hq, d)).astype(np.float32))
        out = torch.empty(B, S, Hq, d, dtype=torch.bfloat16, device="cuda")
        ssd.ssd_branch_attention(to_dev(q), gk, gv, gtable, gprefix, to_dev(parent), out, status=st)
        ref_o, _, afl = oracle.branch_attention(q, kc, vc, table, prefix, parent, Hkv)
        assert afl.tolist() == [0] * B
        np.testing.assert_allclose(out.float().cpu().numpy(), ref_o, atol=2e-2, rtol=0)
        logits = w.fill_step_logits(spec, 3, t)
        u = w.fill_uniforms(3, 0, t, B, S)
        ws = ssd.fill_workspace(B, S, spec.V, spec.dtype, spec.F[t])
        tok = torch.empty(B, S, dtype=torch.int32, device="cuda")
        ssd.ssd_fill_sample(to_dev(logits), spec.V, spec.F[t], spec.C, spec.T, to_dev(u), tok, t=t,
                            payload=payload, status=st, ws=ws)
        rt, _, mg = oracle.fill_sample(logits, spec.V, spec.F[t], spec.C, spec.T, u)
        torch.cuda.synchronize()
        g = tok.cpu().numpy()
        ok = mg >= NEAR_TIE
        np.testing.assert_array_equal(g[ok], rt[ok])
        ref_payload[:, :, t] = g
    assert int(st.item()) == 0
    np.testing.assert_array_equal(gk.cpu().view(torch.int16).numpy().view(np.uint16), kc)
    np.testing.assert_array_equal(gv.cpu().view(torch.int16).numpy().view(np.uint16), vc)
    np.testing.assert_array_equal(payload.cpu().numpy(), ref_payload)

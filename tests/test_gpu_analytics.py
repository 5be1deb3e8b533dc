"""GPU parity of the round analytics (ssd_round_analytics) against the fp64
oracle: acceptance rates, residual masses, the accept-count distribution, the
chance that the bonus lands among each depth's guesses, the exact hit rate
and the expected tokens per round, all within 1e-5 relative."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_vocab_gb300 import binding as ssd
from speculative_decoding_vocab_gb300 import workloads as w

from parity import batched, to_dev

pytestmark = pytest.mark.gpu
RTOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_vocab_gb300 import build
    build.build()
    ssd.load()


def gpu_analytics(inp, T=None, C=None):
    spec = inp.spec
    T = spec.T if T is None else T
    C = spec.C if C is None else C
    B, K = spec.B, spec.K
    f32 = dict(dtype=torch.float32, device="cuda")
    o = dict(alpha=torch.full((B, K), -1.0, **f32), resid_w=torch.full((B, K), -1.0, **f32),
             p_accept=torch.full((B, K + 1), -1.0, **f32),
             hit_mass=torch.full((B, K + 1), -1.0, **f32), hit_rate=torch.full((B,), -1.0, **f32),
             exp_tokens=torch.full((B,), -1.0, **f32))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = ssd.workspace(B, K, spec.V, spec.dtype, spec.F)
    ssd.ssd_round_analytics(to_dev(inp.target), to_dev(inp.draft), spec.V, spec.F, C, T,
                            o["p_accept"], o["hit_rate"], o["exp_tokens"], alpha=o["alpha"],
                            resid_w=o["resid_w"], hit_mass=o["hit_mass"], status=st, ws=ws)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy().astype(np.float64) for k, v in o.items()}
    res["status"] = int(st.item())
    return res


def compare(inp, T=None, C=None, rtol=RTOL):
    spec = inp.spec
    T = spec.T if T is None else T
    C = spec.C if C is None else C
    g = gpu_analytics(inp, T, C)
    ref = batched(lambda t_, d_: oracle.round_analytics(t_, d_, spec.V, spec.F, C, T), spec.B,
                  (inp.target, inp.draft))
    for k in ("alpha", "resid_w", "p_accept", "hit_mass", "hit_rate", "exp_tokens"):
        a, b = g[k], ref[k]
        tol = rtol * np.maximum(np.abs(b), 1e-30)
        if k == "hit_mass":
            # a difference of probabilities: fp32 row statistics (relative
            # error below 1e-6) move it by up to 1e-6 times its terms' size
            tol = tol + 1e-6 * ref["hit_scale"]
        if k == "hit_rate":
            tol = tol + 1e-6 * (ref["p_accept"] * ref["hit_scale"]).sum(axis=1)
        ok = np.abs(a - b) <= tol
        assert ok.all(), (k, np.argwhere(~ok)[:5].tolist(), a[~ok][:5], b[~ok][:5])
    assert g["status"] == 0
    return g, ref


def test_llama3_round_analytics_full():
    inp = w.make_round(w.llama3_round(T=1.0), seed=0)
    g, ref = compare(inp)
    print(f"Llama-3 round: mean alpha {g['alpha'].mean():.4f}, hit rate {g['hit_rate'].mean():.4f}, "
          f"E[tokens] {g['exp_tokens'].mean():.4f}")


@pytest.mark.parametrize("C", [1.0, 0.25])
def test_qwen3_round_analytics_full(C):
    inp = w.make_round(w.qwen3_round(C=C), seed=0)
    g, ref = compare(inp)
    print(f"Qwen-3 C={C}: exact hit rate {g['hit_rate'].mean():.4f}")


def test_tiny_rounds_analytics():
    spec = w.tiny_round()
    parts = [w.make_round(spec, seed=0, rnd=r) for r in range(200)]
    big = w.RoundSpec(**{**spec.__dict__, "B": len(parts)})
    inp = w.RoundInputs(big, np.concatenate([p.target for p in parts]),
                        np.concatenate([p.draft for p in parts]),
                        np.concatenate([p.u_draft for p in parts]),
                        np.concatenate([p.u_acc for p in parts]),
                        np.concatenate([p.u_bonus for p in parts]), None)
    compare(inp)


@pytest.mark.parametrize("dtype,V,pad,K,F,T,C", [
    ("bf16", 70001, 7, 5, (16, 8, 4, 2, 1, 1), 0.7, 0.5),   # ragged tail, C < 1
    ("f32", 37, 3, 3, (3, 2, 1, 1), 1.0, 0.25),            # tail smaller than one vector
    ("f32", 8, 0, 3, (8, 8, 8, 8), 0.8, 0.5),              # F_k = V: every token guessed
    ("bf16", 40000, 0, 0, (5,), 1.0, 1.0),                 # K = 0: one token per round
    ("bf16", 33000, 8, 2, (256, 100, 1), 1.0, 0.5),        # F at its maximum
    ("bf16", 20000, 0, 4, (6, 3, 2, 1, 1), 0.0, 0.5),      # greedy limit
])
def test_analytics_shapes(dtype, V, pad, K, F, T, C):
    spec = w.RoundSpec(B=6, K=K, V=V, dtype=dtype, recipe="gauss", T=T, C=C, F=F,
                       target_sigma=2.0, draft_noise=0.7, row_pad=pad)
    compare(w.make_round(spec, seed=V + K + 3))


def test_analytics_predict_the_sampled_rounds():
    """The analytic hit rate and expected tokens against the same round drawn
    many times on the GPU (ssd_round with fresh uniforms): Monte Carlo within
    5 standard errors."""
    spec = w.RoundSpec(B=1, K=3, V=500, dtype="f32", recipe="gauss", T=1.0, C=0.5,
                       F=(6, 3, 2, 1), target_sigma=1.5, draft_noise=0.8)
    one = w.make_round(spec, seed=9)
    n = 20000
    tgt = np.broadcast_to(one.target, (n,) + one.target.shape[1:]).copy()
    dft = np.broadcast_to(one.draft, (n,) + one.draft.shape[1:]).copy()
    ud, ua, ub = w.round_uniforms(31, 0, n, spec.K)
    big = w.RoundSpec(**{**spec.__dict__, "B": n})
    inp = w.RoundInputs(big, tgt, dft, ud, ua, ub, None)
    from parity import gpu_round
    g = gpu_round(inp)
    hits = g["slot"] >= 0
    toks = g["accept_len"] + 1
    an = gpu_analytics(one)
    h, e = an["hit_rate"][0], an["exp_tokens"][0]
    assert abs(hits.mean() - h) < 5 * np.sqrt(h * (1 - h) / n)
    assert abs(toks.mean() - e) < 5 * toks.std() / np.sqrt(n)

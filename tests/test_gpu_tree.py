"""GPU parity of token-tree verification (ssd_tree_verify) against the
oracle: the walk (accept counts, accepted node paths, emitted tokens) and the
bonus bit-exact unless one of the sequence's decisions is a near-tie (its
uniform within 1e-6 of the threshold in the oracle's exact arithmetic), the
residual mass within 1e-5 relative; every cluster size the vocabulary sizes
select (1, 3, 4 and 8 CTAs per sequence), ragged rows, T = 0, trees without
nodes, flags and argument errors."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_vocab_gb300 import binding as ssd
from speculative_decoding_vocab_gb300 import workloads as w

from parity import NEAR_TIE, batched, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_vocab_gb300 import build
    build.build()
    ssd.load()


def draw_children(spec, draft, parent, seed):
    """Each node's token drawn from the draft's q at its parent (the oracle's
    softmax, numpy inverse CDF): the children a draft would propose."""
    rng = np.random.default_rng(seed)
    B, N = draft.shape[0], len(parent)
    z = draft if spec.dtype == "f32" else w.bf16_bits_to_f32(draft)
    tok = np.zeros((B, N), np.int32)
    for b in range(B):
        for m in range(N):
            q = oracle.softmax(z[b, parent[m] + 1, :spec.V].astype(np.float64), spec.T)
            cdf = np.cumsum(q)
            tok[b, m] = min(int(np.searchsorted(cdf, rng.random() * cdf[-1], side="right")), spec.V - 1)
    return tok


def inputs(spec, seed, pad=0):
    tgt, dft = w.tree_logits(spec, seed)
    if pad:
        tgt = np.concatenate([tgt, np.zeros(tgt.shape[:2] + (pad,), tgt.dtype)], axis=2)
        dft = np.concatenate([dft, np.zeros(dft.shape[:2] + (pad,), dft.dtype)], axis=2)
    parent1 = w.tree_shape(spec.branching)
    tok = draw_children(spec, dft, parent1, seed + 1)
    par = np.broadcast_to(parent1, (spec.B, len(parent1))).copy()
    ua, ub = w.tree_uniforms(seed, 0, spec.B, len(parent1))
    return tgt, dft, par, tok, ua, ub


def gpu_tree(spec, tgt, dft, par, tok, ua, ub):
    B, N = par.shape
    i32 = dict(dtype=torch.int32, device="cuda")
    o = dict(accept_len=torch.full((B,), -7, **i32), path=torch.full((B, N), -7, **i32),
             bonus=torch.full((B,), -7, **i32), out_tokens=torch.full((B, N + 1), -7, **i32),
             resid_mass=torch.full((B,), -1.0, dtype=torch.float32, device="cuda"),
             status=torch.zeros(1, **i32))
    ssd.ssd_tree_verify(to_dev(tgt), to_dev(dft), spec.V, spec.T, to_dev(par), to_dev(tok),
                        to_dev(ua), to_dev(ub), o["accept_len"], o["path"], o["bonus"],
                        out_tokens=o["out_tokens"], resid_mass=o["resid_mass"], status=o["status"])
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in o.items()}


def compare(spec, tgt, dft, par, tok, ua, ub, expect_flags=0):
    g = gpu_tree(spec, tgt, dft, par, tok, ua, ub)
    assert int(g["status"][0]) == expect_flags
    B, N = par.shape
    r = batched(lambda t_, d_, p_, k_, a_, b_: oracle.tree_verify(t_, d_, spec.V, spec.T, p_, k_, a_, b_),
                B, (tgt, dft, par, tok, ua, ub))
    near = (r["acc_margin"] < NEAR_TIE).any(axis=1) | (r["bonus_margin"] < NEAR_TIE)
    ok = ~near
    assert ok.mean() >= 0.75, ok.mean()
    np.testing.assert_array_equal(g["accept_len"][ok], r["accept_len"][ok])
    np.testing.assert_array_equal(g["path"][ok], r["path"][ok])
    np.testing.assert_array_equal(g["bonus"][ok], r["bonus"][ok])
    for b in np.nonzero(ok)[0]:
        L = r["accept_len"][b]
        want = [int(tok[b, m]) for m in r["path"][b, :L]] + [int(r["bonus"][b])] + [-1] * (N - L)
        assert g["out_tokens"][b].tolist() == want
    np.testing.assert_allclose(g["resid_mass"][ok], r["resid_mass"][ok], rtol=1e-5, atol=0)
    return g, r, int(near.sum())


@pytest.mark.parametrize("T", [1.0, 0.6, 0.0])
def test_tree_tiny(T):
    spec = dataclasses.replace(w.tiny_tree(), T=T, B=24)
    g, r, _ = compare(spec, *inputs(spec, 3))
    assert (r["accept_len"] > 0).any() and (r["accept_len"] == 0).any()


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_tree_children_at_target_argmax(T):
    """Even children carry the target's argmax at their parent, odd ones the
    token after it: at T = 0 every even child is accepted whatever the draft
    prefers, so each walk reaches the deepest level."""
    spec = w.TreeSpec(B=6, V=3000, dtype="f32", T=T, branching=(2, 2), recipe="gauss",
                      draft_noise=0.8, name="argmax-children")
    tgt, dft = w.tree_logits(spec, 21)
    parent1 = w.tree_shape(spec.branching)
    N = len(parent1)
    am = tgt.argmax(axis=2)[:, parent1 + 1]
    tok = np.ascontiguousarray(np.where(np.arange(N)[None, :] % 2 == 0, am, (am + 1) % spec.V),
                               dtype=np.int32)
    par = np.broadcast_to(parent1, (spec.B, N)).copy()
    ua, ub = w.tree_uniforms(21, 0, spec.B, N)
    g, r, _ = compare(spec, tgt, dft, par, tok, ua, ub)
    if T == 0.0:
        assert (r["accept_len"] == 2).all()


def test_tree_chain_of_max_nodes_greedy():
    """A chain of 256 nodes (the largest tree) whose tokens are the target's
    argmax at T = 0: every walk goes the whole way down, 256 nodes deep."""
    B, N, V = 2, 256, 640
    spec = w.TreeSpec(B=B, V=V, dtype="f32", T=0.0, branching=(1,) * N, recipe="gauss",
                      draft_noise=0.8, name="chain256")
    tgt, dft = w.tree_logits(spec, 23)
    parent1 = np.arange(-1, N - 1, dtype=np.int32)
    assert np.array_equal(parent1, w.tree_shape(spec.branching))
    tok = np.ascontiguousarray(tgt.argmax(axis=2)[:, :N], dtype=np.int32)
    par = np.broadcast_to(parent1, (B, N)).copy()
    ua, ub = w.tree_uniforms(23, 0, B, N)
    g, r, _ = compare(spec, tgt, dft, par, tok, ua, ub)
    assert (g["accept_len"] == N).all()


def test_tree_binary_254_nodes():
    """A binary tree seven levels deep (254 nodes), children drawn from the draft."""
    spec = w.TreeSpec(B=4, V=700, dtype="f32", T=1.0, branching=(2,) * 7, recipe="gauss",
                      draft_noise=0.6, name="binary254")
    compare(spec, *inputs(spec, 25))


def test_tree_llama3_full_batch():
    """The 28-node tree over the Llama-3 vocabulary (4 CTAs per sequence), all
    32 sequences."""
    spec = w.llama3_tree()
    g, r, _ = compare(spec, *inputs(spec, 5))
    assert r["accept_len"].mean() > 0.5


def test_tree_ragged_vocabulary_three_ctas():
    """V = 70001 bf16 (a partial last vector; 3 CTAs per sequence), rows padded."""
    spec = dataclasses.replace(w.llama3_tree(B=6), V=70001, name="ragged")
    compare(spec, *inputs(spec, 7, pad=7))


def test_tree_eight_ctas_fp32():
    """V = 131072 fp32 (512 KiB rows: the largest, 8 CTAs per sequence)."""
    spec = w.TreeSpec(B=3, V=131072, dtype="f32", T=1.0, branching=(2, 1), recipe="gauss",
                      draft_noise=0.8, name="f32-8ctas")
    compare(spec, *inputs(spec, 9))


def test_tree_small_vocabulary_and_wide_root():
    spec = w.TreeSpec(B=40, V=8, dtype="f32", T=1.0, branching=(6, 3), recipe="gauss",
                      draft_noise=1.0, name="V8")
    compare(spec, *inputs(spec, 11))


def test_tree_without_nodes():
    """N = 0: the bonus is drawn from the root's p."""
    spec = dataclasses.replace(w.tiny_tree(), B=5)
    tgt, dft, _, _, _, ub = inputs(spec, 13)
    tgt, dft = np.ascontiguousarray(tgt[:, :1]), np.ascontiguousarray(dft[:, :1])
    par = np.zeros((spec.B, 0), np.int32)
    g, r, _ = compare(spec, tgt, dft, par, par.copy(), np.zeros((spec.B, 0), np.float32), ub)
    assert (g["accept_len"] == 0).all()


def test_tree_flags():
    spec = dataclasses.replace(w.tiny_tree(), B=4)
    tgt, dft, par, tok, ua, ub = inputs(spec, 15)
    par[1, 4] = 9        # after node 4: nobody's child
    tok[2, 0] = spec.V   # outside the vocabulary: skipped
    compare(spec, tgt, dft, par, tok, ua, ub, expect_flags=ssd.FLAG_BAD_TREE | ssd.FLAG_BAD_TOKEN)


def test_tree_argument_checks():
    i32 = dict(dtype=torch.int32, device="cuda")
    lg = torch.zeros(1, 258, 16, device="cuda")
    z = torch.zeros(1, 257, **i32)
    o = [torch.zeros(1, **i32), torch.zeros(1, 257, **i32), torch.zeros(1, **i32)]
    st = torch.zeros(1, **i32)
    with pytest.raises(ssd.SSDError):  # more than 256 nodes
        ssd.ssd_tree_verify(lg, lg, 16, 1.0, z, z, z.float(), torch.zeros(1, device="cuda"), *o,
                            status=st)
    big = torch.zeros(1, 2, 131080, device="cuda")
    z1 = torch.zeros(1, 1, **i32)
    with pytest.raises(ssd.SSDError):  # rows above 512 KiB
        ssd.ssd_tree_verify(big, big, 131080, 1.0, z1, z1, z1.float(), torch.zeros(1, device="cuda"),
                            o[0], z1, o[2], status=st)

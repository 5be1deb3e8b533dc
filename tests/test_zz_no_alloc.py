"""The no-allocation verification entry point.

Some callers cannot allocate device memory themselves (a plugin inside another
framework that owns every device allocation, or a plain C program with no
allocator of its own), so ``ssd_verify_noalloc`` runs verification on a fixed
scratch array inside the library instead of a caller workspace.  This test
calls it through the C ABI twice in a row and checks each result against the
workspace entry point ``ssd_verify`` on the same inputs, and both against the
fp64 oracle, with the tolerances the other parity tests use (integers exact,
probabilities and residual masses within 1e-5 relative).  It lives in its own
file, collected last, and passes alone or after the other tests.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_vocab_gb300 import binding as ssd
from speculative_decoding_vocab_gb300 import workloads as w

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_vocab_gb300 import build
    build.build()
    ssd.load()


def _rel_ok(a, b, rtol=1e-5):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.all(np.abs(a - b) <= rtol * np.maximum(np.abs(b), 1e-30))


def _verify(entry, inp, d):
    spec = inp.spec
    B, K, V = spec.B, spec.K, spec.V
    dev = "cuda"
    i32 = dict(dtype=torch.int32, device=dev)
    out = dict(accept_len=torch.full((B,), -9, **i32), out_tokens=torch.full((B, K + 1), -9, **i32),
               bonus=torch.full((B,), -9, **i32),
               accept_prob=torch.zeros(B, K, dtype=torch.float32, device=dev),
               resid_mass=torch.zeros(B, dtype=torch.float32, device=dev),
               near_ties=torch.zeros(1, **i32), status=torch.zeros(1, **i32))
    args = (ssd.tensor(inp.target), ssd.tensor(inp.draft), V, spec.F, spec.C, spec.T, d,
            ssd.tensor(inp.u_acc), ssd.tensor(inp.u_bonus), out["accept_len"], out["out_tokens"],
            out["bonus"])
    kw = dict(accept_prob=out["accept_prob"], resid_mass=out["resid_mass"], status=out["status"],
              near_ties=out["near_ties"])
    if entry == "workspace":
        ssd.ssd_verify(*args, ws=ssd.workspace(B, K, V, spec.dtype, spec.F), **kw)
    else:
        ssd.ssd_verify_noalloc(*args, **kw)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    for call, spec in enumerate([w.llama3_round(T=1.0, B=8),
                                 w.RoundSpec(B=5, K=3, V=70001, dtype="bf16", recipe="zipf", T=0.6,
                                             C=0.5, F=(9, 4, 2, 1), draft_noise=1.5, row_pad=7)]):
        inp = w.make_round(spec, seed=40 + call)
        assert ssd.ssd_workspace_size(spec.B, spec.K, spec.V, spec.dtype, spec.F) <= \
            ssd.ssd_verify_noalloc_max_bytes()
        # the draft tokens to verify: the draft's own argmax chain with some perturbed
        d = np.argmax(w.bf16_bits_to_f32(inp.draft[:, :spec.K, :spec.V]), axis=-1).astype(np.int32)
        d[::2, 0] = (d[::2, 0] + 7) % spec.V
        dd = ssd.tensor(d)
        ref = _verify("workspace", inp, dd)
        got = _verify("static", inp, dd)
        assert got["status"][0] == 0 and ref["status"][0] == 0, call
        for k in ("accept_len", "out_tokens", "bonus", "near_ties"):
            assert np.array_equal(got[k], ref[k]), (call, k)
        assert _rel_ok(got["accept_prob"], ref["accept_prob"]), call
        assert _rel_ok(got["resid_mass"], ref["resid_mass"]), call
        # and against the oracle (no decision of these seeds differs within a near-tie)
        ov = oracle.verify(inp.target, inp.draft, spec.V, spec.F, spec.C, spec.T, d, inp.u_acc,
                           inp.u_bonus)
        assert np.array_equal(got["accept_len"], ov["accept_len"]), call
        assert np.array_equal(got["out_tokens"], ov["out_tokens"]), call
        assert _rel_ok(got["accept_prob"], ov["accept_prob"]), call
        assert _rel_ok(got["resid_mass"], ov["resid_mass"]), call
        # the near-ties counted: those of the oracle's exact margins
        o_nt = int((ov["acc_margin"] < 1e-6).sum() + (ov["bonus_margin"] < 1e-6).sum())
        assert abs(int(got["near_ties"][0]) - o_nt) <= 2, (call, got["near_ties"][0], o_nt)


def test_noalloc_rejects_batches_beyond_its_scratch():
    spec = w.llama3_round(T=1.0, B=2)
    need_b = 1
    while ssd.ssd_workspace_size(need_b, spec.K, spec.V, "bf16", spec.F) <= ssd.ssd_verify_noalloc_max_bytes():
        need_b *= 2
    B = need_b
    # only shapes are checked before the refusal; no memory of that size is touched
    dev = "cuda"
    tgt = torch.zeros(1, spec.K + 1, spec.V, dtype=torch.bfloat16, device=dev).expand(B, -1, -1)
    i32 = dict(dtype=torch.int32, device=dev)
    st = torch.zeros(1, **i32)
    with pytest.raises(ssd.SSDError) as e:
        ssd.ssd_verify_noalloc(tgt, tgt, spec.V, spec.F, 1.0, 1.0, torch.zeros(B, spec.K, **i32),
                               torch.zeros(B, spec.K, device=dev), torch.zeros(B, device=dev),
                               torch.zeros(B, **i32), torch.zeros(B, spec.K + 1, **i32),
                               torch.zeros(B, **i32), status=st)
    assert e.value.code == ssd.SSD_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int(st.item()) == 0  # nothing was launched

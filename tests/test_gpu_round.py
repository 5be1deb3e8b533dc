"""GPU parity of the speculation-round calls against the fp64 oracle.

Every test drives the CUDA library through its C ABI (ctypes binding) on seeded
inputs and compares element by element with the oracle (rules in parity.py).
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_vocab_gb300 import binding as ssd
from speculative_decoding_vocab_gb300 import workloads as w

from parity import Report, compare_round, gpu_round, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_vocab_gb300 import build
    build.build()
    ssd.load()


def _stack_rounds(spec, nrounds, seed=0):
    """nrounds independent B=1 rounds of ``spec`` stacked as one batch; each row
    keeps its own round's logits and uniforms."""
    parts = [w.make_round(spec, seed=seed, rnd=r) for r in range(nrounds)]
    big = w.RoundSpec(**{**spec.__dict__, "B": nrounds})
    return w.RoundInputs(big, np.concatenate([p.target for p in parts]),
                         np.concatenate([p.draft for p in parts]),
                         np.concatenate([p.u_draft for p in parts]),
                         np.concatenate([p.u_acc for p in parts]),
                         np.concatenate([p.u_bonus for p in parts]),
                         np.concatenate([p.payload for p in parts]))


# ---------------------------------------------------------------------------
# the workloads
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fused", [True, False])
def test_tiny_round_1000_rounds(fused):
    inp = _stack_rounds(w.tiny_round(), 1000)
    g = gpu_round(inp, fused=fused)
    rep = compare_round(inp, g)
    assert g["status"][0] == 0
    print(rep)


def test_tiny_round_single_launches():
    spec = w.tiny_round()
    rep = Report()
    for r in range(20):
        inp = w.make_round(spec, seed=0, rnd=r)
        compare_round(inp, gpu_round(inp), report=rep)
    assert rep.compared == 20


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_llama3_round_full(T):
    inp = w.make_round(w.llama3_round(T=T), seed=0)
    g = gpu_round(inp)
    rep = compare_round(inp, g)
    print(rep, "hits", int(g["hits"][0]))


@pytest.mark.parametrize("C", [1.0, 0.5, 0.25])
def test_qwen3_round_full(C):
    """All 256 sequences of the Qwen-3 round against the oracle, per C."""
    spec = w.qwen3_round(C=C)
    inp = w.make_round(spec, seed=0)
    g = gpu_round(inp)
    rep = compare_round(inp, g)
    assert rep.compared == spec.B and g["status"][0] == 0
    print(rep, f"C={C} hit rate {int(g['hits'][0]) / spec.B:.4f}")


def test_llama3_round_at_scale_full():
    """All 64 sequences of the round that accompanies verify-shaped attention."""
    spec = w.llama3_round_at_scale()
    inp = w.make_round(spec, seed=0)
    g = gpu_round(inp)
    rep = compare_round(inp, g)
    assert rep.compared == spec.B and g["status"][0] == 0
    print(rep, "hits", int(g["hits"][0]))


def test_separate_calls_equal_fused_call():
    inp = w.make_round(w.llama3_round(T=1.0, B=8), seed=3)
    a = gpu_round(inp, fused=True)
    b = gpu_round(inp, fused=False)
    for k in ("d", "qd", "accept_len", "out_tokens", "bonus", "accept_prob", "resid_mass", "guess",
              "guess_q", "slot", "next_tokens", "hits"):
        assert np.array_equal(a[k], b[k]), k


# ---------------------------------------------------------------------------
# shapes, ragged tails and degenerate cases
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype,V,pad,K,F", [
    ("bf16", 70001, 7, 5, (16, 8, 4, 2, 1, 1)),     # several chunks and a ragged tail
    ("f32", 37, 3, 3, (3, 2, 1, 1)),               # tail smaller than one vector
    ("f32", 8, 0, 3, (8, 8, 8, 8)),                # F_k = V
    ("bf16", 8, 0, 2, (8, 1, 8)),
    ("bf16", 40000, 0, 0, (5,)),                   # K = 0: only the bonus draw
    ("f32", 9000, 4, 16, tuple([2] * 17)),         # K = 16
    ("bf16", 33000, 8, 2, (256, 100, 1)),          # F at its maximum
])
@pytest.mark.parametrize("T", [0.0, 0.7])
def test_shapes(dtype, V, pad, K, F, T):
    spec = w.RoundSpec(B=5, K=K, V=V, dtype=dtype, recipe="gauss", T=T, C=0.5, F=F,
                       target_sigma=2.0, draft_noise=0.7, row_pad=pad)
    inp = w.make_round(spec, seed=V + K)
    compare_round(inp, gpu_round(inp))


@pytest.mark.parametrize("dtype,V", [("bf16", 1 << 21), ("f32", 1 << 20)])
def test_largest_rows(dtype, V):
    """Rows of the largest supported size, 4 MiB (1024 segments of 4 KiB): every
    sequence against the oracle."""
    spec = w.RoundSpec(B=2, K=2, V=V, dtype=dtype, recipe="gauss", T=0.7, C=0.5, F=(16, 4, 1),
                       target_sigma=2.0, draft_noise=0.7, row_pad=0)
    inp = w.make_round(spec, seed=21)
    compare_round(inp, gpu_round(inp))


def test_zero_batch_is_a_noop():
    spec = w.RoundSpec(B=0, K=3, V=100, dtype="f32", recipe="gauss", F=(2, 1, 1, 1))
    inp = w.make_round(spec)
    g = gpu_round(inp)
    assert g["hits"][0] == 0 and g["status"][0] == 0


def test_all_equal_logits_ties():
    """Every logit equal: top-F and argmax break ties by the lower index; the
    pair merge's top-F overflows its candidate buffers and takes its tie
    fallback (one winner per sweep)."""
    spec = w.RoundSpec(B=3, K=3, V=50000, dtype="bf16", recipe="gauss", T=1.0, C=0.5,
                       F=(40, 20, 3, 1))
    inp = w.make_round(spec, seed=1)
    inp.target[...] = w.f32_to_bf16_bits(np.float32(0.5))
    inp.draft[...] = w.f32_to_bf16_bits(np.float32(0.5))
    inp.draft[1, :, 777] = w.f32_to_bf16_bits(np.float32(0.75))
    for T in (0.0, 1.0):
        compare_round(inp, gpu_round(inp, T=T), T=T)


def test_neg_inf_logits():
    spec = w.RoundSpec(B=4, K=3, V=20000, dtype="f32", recipe="gauss", T=1.0, C=0.25,
                       F=(6, 3, 2, 1))
    inp = w.make_round(spec, seed=2)
    rng = np.random.default_rng(0)
    mask = rng.random(inp.target.shape) < 0.3
    inp.target[mask] = -np.inf
    inp.draft[rng.random(inp.draft.shape) < 0.3] = -np.inf
    compare_round(inp, gpu_round(inp))


def test_bad_token_and_zero_residual_flags():
    spec = w.RoundSpec(B=6, K=3, V=3000, dtype="f32", recipe="gauss", T=1.0, C=1.0,
                       F=(2, 1, 1, 1), draft_noise=0.0)
    inp = w.make_round(spec, seed=5)
    dev = "cuda"
    B, K, V = spec.B, spec.K, spec.V
    d = np.zeros((B, K), np.int32)
    d[:, 1] = V + 5  # invalid at position 2 -> rejected there; p == q so the residual is empty
    i32 = dict(dtype=torch.int32, device=dev)
    acc = torch.empty(B, **i32)
    out = torch.empty(B, K + 1, **i32)
    bon = torch.empty(B, **i32)
    ap = torch.empty(B, K, dtype=torch.float32, device=dev)
    rm = torch.empty(B, dtype=torch.float32, device=dev)
    st = torch.zeros(1, **i32)
    ssd.ssd_verify(to_dev(inp.target), to_dev(inp.draft), V, spec.F, 1.0, 1.0, to_dev(d),
                   to_dev(inp.u_acc), to_dev(inp.u_bonus), acc, out, bon, ap, rm, status=st,
                   ws=ssd.workspace(B, K, V, "f32", spec.F))
    torch.cuda.synchronize()
    ov = oracle.verify(inp.target, inp.draft, V, spec.F, 1.0, 1.0, d, inp.u_acc, inp.u_bonus)
    assert np.array_equal(acc.cpu().numpy(), ov["accept_len"])
    assert np.array_equal(out.cpu().numpy(), ov["out_tokens"])
    flags = int(st.item())
    assert flags & ssd.FLAG_BAD_TOKEN and flags & ssd.FLAG_ZERO_RESIDUAL
    assert np.all(ov["flags"] & oracle.FLAG_ZERO_RESIDUAL)
    assert np.all(ap.cpu().numpy()[:, 1] == 0)


def test_lookup_bad_outcome_flag():
    B, K = 50, 4
    F = (4, 2, 1, 1, 1)
    rng = np.random.default_rng(3)
    guess = rng.integers(0, 20, size=(B, sum(F))).astype(np.int32)
    payload = rng.integers(0, 1000, size=(B, sum(F), K)).astype(np.int32)
    a = rng.integers(-1, K + 2, size=B).astype(np.int32)
    b = rng.integers(0, 20, size=B).astype(np.int32)
    i32 = dict(dtype=torch.int32, device="cuda")
    slot = torch.empty(B, **i32)
    nt = torch.empty(B, K, **i32)
    hits = torch.empty(1, **i32)
    st = torch.zeros(1, **i32)
    ssd.ssd_cache_lookup(to_dev(guess), to_dev(payload), K, F, to_dev(a), to_dev(b), slot, nt, hits,
                         status=st)
    torch.cuda.synchronize()
    ol = oracle.lookup(guess, payload, K, F, a, b)
    assert np.array_equal(slot.cpu().numpy(), ol["slot"])
    assert np.array_equal(nt.cpu().numpy(), ol["next_tokens"])
    assert int(hits.item()) == ol["hits"]
    assert int(st.item()) & ssd.FLAG_BAD_OUTCOME


# ---------------------------------------------------------------------------
# host-side argument errors: nothing is launched, the status word stays 0
# ---------------------------------------------------------------------------
def test_argument_errors():
    spec = w.RoundSpec(B=2, K=2, V=1000, dtype="f32", recipe="gauss", F=(2, 1, 1))
    inp = w.make_round(spec)
    dev = "cuda"
    i32 = dict(dtype=torch.int32, device=dev)
    st = torch.zeros(1, **i32)
    d = torch.empty(2, 2, **i32)
    ws = ssd.workspace(2, 2, 1000, "f32", spec.F)
    dft = to_dev(inp.draft)
    ud = to_dev(inp.u_draft)
    with pytest.raises(ssd.SSDError) as e:  # C outside (0, 1]
        ssd.ssd_saguaro_sample(dft, 1000, spec.F, 0.0, 1.0, ud, d, status=st, ws=ws)
    assert e.value.code == ssd.SSD_ERR_INVALID_ARG
    with pytest.raises(ssd.SSDError) as e:  # F_k > V
        ssd.ssd_saguaro_sample(dft, 1000, (2000, 1, 1), 0.5, 1.0, ud, d, status=st, ws=ws)
    assert e.value.code == ssd.SSD_ERR_UNSUPPORTED
    with pytest.raises(ssd.SSDError) as e:  # workspace too small
        ssd.ssd_saguaro_sample(dft, 1000, spec.F, 0.5, 1.0, ud, d, status=st, ws=ws[:16])
    assert e.value.code == ssd.SSD_ERR_WORKSPACE
    big = torch.zeros(2, 3, 1003, dtype=torch.float32, device=dev)[:, :, 1:]  # 4-byte offset
    with pytest.raises(ssd.SSDError) as e:
        ssd.ssd_saguaro_sample(big, 1000, spec.F, 0.5, 1.0, ud, d, status=st, ws=ws)
    assert e.value.code == ssd.SSD_ERR_UNSUPPORTED
    with pytest.raises(ssd.SSDError) as e:  # negative temperature
        ssd.ssd_saguaro_sample(dft, 1000, spec.F, 0.5, -1.0, ud, d, status=st, ws=ws)
    assert e.value.code == ssd.SSD_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def test_one_workspace_across_calls_of_every_kind():
    """One workspace (filled with 0xFF bytes first) serves verification calls of
    several shapes, temperatures and C, with analytics, sampling and
    separate-call rounds in between: every result equals the oracle's, so no
    call leaves a stale record or ready word for the next."""
    import dataclasses
    a = w.RoundSpec(B=6, K=4, V=4096, dtype="f32", recipe="gauss", T=1.0, C=1.0,
                    F=(4, 2, 1, 1, 1), draft_noise=0.5, name="reuse-a")
    b = dataclasses.replace(a, B=3, K=2, F=(3, 2, 1), name="reuse-b")
    c = dataclasses.replace(a, V=5000, dtype="bf16", recipe="zipf", C=0.5, draft_noise=1.0,
                            name="reuse-c")
    n = max(ssd.ssd_workspace_size(s.B, s.K, s.V, s.dtype, s.F) for s in (a, b, c))
    ws = torch.full((n,), 255, dtype=torch.uint8, device="cuda")
    rep = Report()
    ia, ib, ic = w.make_round(a, seed=31), w.make_round(b, seed=32), w.make_round(c, seed=33)
    for step, (inp, kw) in enumerate([(ia, {}), (ib, {}), (ia, {"fused": False}), (ic, {}),
                                      (ia, {"T": 0.0}), (ib, {"fused": False}), (ic, {"T": 0.0}),
                                      (ia, {})]):
        g = gpu_round(inp, ws=ws, **kw)
        compare_round(inp, g, T=kw.get("T"), report=rep)
        if step == 3:  # an analytics call on the same workspace in between
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            f32 = dict(dtype=torch.float32, device="cuda")
            ssd.ssd_round_analytics(to_dev(ib.target), to_dev(ib.draft), b.V, b.F, b.C, b.T,
                                    torch.empty(b.B, b.K + 1, **f32), torch.empty(b.B, **f32),
                                    torch.empty(b.B, **f32), status=st, ws=ws)
            torch.cuda.synchronize()
            assert int(st.item()) == 0
    assert rep.compared == 6 + 3 + 6 + 6 + 6 + 3 + 6 + 6


def test_pipelined_rounds_back_to_back():
    """Rounds of independent batches with ssd_round_pipelined, launched back to
    back without a synchronize so that each statistics pass overlaps the
    previous round's tail: every round equals the oracle (and so ssd_round)."""
    from parity import collect_round, enqueue_round, prepare_round
    spec = w.llama3_round(T=1.0)
    inps = [w.make_round(spec, seed=40 + i) for i in range(4)]
    small = w.RoundSpec(B=5, K=3, V=7000, dtype="bf16", recipe="zipf", T=0.7, C=0.5,
                        F=(3, 2, 1, 1), draft_noise=1.0, name="pipelined-small")
    inps += [w.make_round(small, seed=50 + i) for i in range(3)]
    # every buffer is ready before the first round: a pipelined round may start
    # before the kernel enqueued just before it has finished
    prepared = [prepare_round(inp) for inp in inps]
    torch.cuda.synchronize()
    launched = [enqueue_round(inp, o, pipelined=True) for inp, o in zip(inps, prepared)]
    torch.cuda.synchronize()
    rep = Report()
    for inp, o in zip(inps, launched):
        g = collect_round(o)
        assert g["status"][0] == 0
        compare_round(inp, g, report=rep)
    assert rep.compared == 4 * 32 + 3 * 5


def test_rounds_on_several_streams():
    """Independent rounds issued round-robin on four streams, pipelined on each
    (the bench's schedule), so that rounds of different streams run at once:
    every round equals the oracle."""
    from parity import collect_round, enqueue_round, prepare_round
    spec = w.llama3_round(T=1.0)
    inps = [w.make_round(spec, seed=60 + i) for i in range(6)]
    small = w.RoundSpec(B=7, K=4, V=9000, dtype="bf16", recipe="zipf", T=1.0, C=0.25,
                        F=(4, 2, 1, 1, 1), draft_noise=1.0, name="streams-small")
    inps += [w.make_round(small, seed=70 + i) for i in range(6)]
    prepared = [prepare_round(inp) for inp in inps]
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    streams = [torch.cuda.Stream() for _ in range(4)]
    for st in streams:
        st.wait_stream(cur)
    launched = []
    for q, (inp, o) in enumerate(zip(inps, prepared)):
        with torch.cuda.stream(streams[q % 4]):
            launched.append(enqueue_round(inp, o, pipelined=True))
    for st in streams:
        cur.wait_stream(st)
    torch.cuda.synchronize()
    rep = Report()
    for inp, o in zip(inps, launched):
        g = collect_round(o)
        assert g["status"][0] == 0
        compare_round(inp, g, report=rep)
    assert rep.compared == 6 * 32 + 6 * 7

"""GPU parity of the miss fallback against the oracle: the n-gram backup
(ssd_ngram_backup; bit-exact proposals and match positions) and the batch
plan (ssd_fallback_plan; fp64 within 1e-12 relative, the same choice)."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_vocab_gb300 import binding as ssd
from speculative_decoding_vocab_gb300 import workloads as w

pytestmark = pytest.mark.gpu
CHUNK = 4096  # candidate positions one scan pass covers


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_vocab_gb300 import build
    build.build()
    ssd.load()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_backup(hist, hist_len, n, K, V, slot, u_rand, plan_best=None, random_option=-1,
               use_slot=True):
    B = u_rand.shape[0]
    nxt = torch.full((B, K), -7, dtype=torch.int32, device="cuda")
    mp = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ssd.ssd_ngram_backup(None if hist is None else dev(hist),
                         None if hist_len is None else dev(hist_len), n, K, V, dev(u_rand), nxt,
                         slot=dev(slot) if use_slot else None, match_pos=mp,
                         plan_best=plan_best, random_option=random_option, status=st)
    torch.cuda.synchronize()
    return nxt.cpu().numpy(), mp.cpu().numpy(), int(st.item())


def check_backup(h, n=None, K=None, use_slot=True):
    sp = h.spec
    n = sp.n if n is None else n
    K = sp.K if K is None else K
    u = np.ascontiguousarray(h.u_rand[:, :K]) if K <= h.u_rand.shape[1] else \
        w.backup_uniforms(5, 0, sp.B, K)
    slot = h.slot if use_slot else np.full(sp.B, -1, np.int32)
    nx, mp, st = gpu_backup(h.hist, h.hist_len, n, K, sp.V, h.slot, u, use_slot=use_slot)
    ref = np.full((sp.B, K), -7, np.int32)
    rnx, rmp = oracle.ngram_backup(h.hist, h.hist_len, n, K, sp.V, slot, u, next_tokens=ref)
    assert st == 0
    np.testing.assert_array_equal(mp, rmp)
    np.testing.assert_array_equal(nx, rnx)
    return rmp


@pytest.mark.parametrize("n", [0, 1, 2, 3, 5])
def test_backup_tiny(n):
    h = w.make_histories(w.tiny_histories(), seed=3)
    mp = check_backup(h, n=n)
    if n in (1, 2):
        assert (mp >= 0).any() and (mp == -1).any() and (mp == -2).any()


def test_backup_every_row_missed_long_proposal():
    h = w.make_histories(w.tiny_histories(), seed=4)
    check_backup(h, K=300, use_slot=False)


def test_backup_qwen3_full_size():
    h = w.make_histories(w.qwen3_histories(), seed=1)
    mp = check_backup(h)
    assert (mp >= 0).any() and (mp == -1).any()


def test_backup_multi_chunk_scan_and_ragged_tail():
    """The only earlier occurrence sits at position 0, several scan chunks and a
    ragged tail below the suffix; a decoy shares the first token only."""
    L = 3 * CHUNK + 123
    rng = np.random.default_rng(9)
    hist = (rng.integers(10, 1000, size=(4, L + 5))).astype(np.int32)
    lens = np.array([L, L, L - 1, 5], np.int32)
    for b in range(3):
        hist[b, :3] = [1, 2, 3]
        hist[b, lens[b] - 3:lens[b]] = [1, 2, 3]
        hist[b, 500:503] = [1, 2, 4]   # first token matches, the rest does not
    hist[3, :5] = [1, 2, 3, 1, 2]        # L = 5, n = 3: the suffix (3, 1, 2) is new
    hist[1, 7000:7003] = [1, 2, 3]       # a later occurrence wins
    K = 6
    u = w.backup_uniforms(2, 0, 4, K)
    slot = np.full(4, -1, np.int32)
    nx, mp, st = gpu_backup(hist, lens, 3, K, 1000, slot, u)
    rnx, rmp = oracle.ngram_backup(hist, lens, 3, K, 1000, slot, u)
    assert st == 0
    assert rmp.tolist() == [0, 7000, 0, -1]
    np.testing.assert_array_equal(mp, rmp)
    np.testing.assert_array_equal(nx, rnx)


def test_backup_policy_gate_skips_search():
    """plan_best == random_option: the random-token backup alone."""
    h = w.make_histories(w.tiny_histories(), seed=3)
    sp = h.spec
    best = torch.tensor([1], dtype=torch.int32, device="cuda")
    nx, mp, st = gpu_backup(h.hist, h.hist_len, sp.n, sp.K, sp.V, h.slot, h.u_rand,
                            plan_best=best, random_option=1)
    rnx, rmp = oracle.ngram_backup(h.hist, h.hist_len, 0, sp.K, sp.V, h.slot, h.u_rand,
                                   next_tokens=np.full((sp.B, sp.K), -7, np.int32))
    np.testing.assert_array_equal(nx, rnx)
    np.testing.assert_array_equal(mp, rmp)
    # another option: the search runs
    nx, mp, _ = gpu_backup(h.hist, h.hist_len, sp.n, sp.K, sp.V, h.slot, h.u_rand,
                           plan_best=best, random_option=0)
    assert (mp >= 0).any()


def test_backup_bad_history_and_token_flags():
    # row 0: suffix (4) last occurs earlier at 2, so h[3] = 77 (outside [0, 10))
    # is proposed: it is replaced by the random token floor(0.5 * 10) = 5.
    # row 1: a length past the row capacity counts as 0: random tokens only.
    hist = np.array([[4, 9, 4, 77, 4], [1, 2, 1, 2, 1]], np.int32)
    lens = np.array([5, 6], np.int32)
    u = np.array([[0.5, 0.25], [0.5, 0.75]], np.float32)
    nx, mp, st = gpu_backup(hist, lens, 1, 2, 10, np.array([-1, -1], np.int32), u)
    assert st == (ssd.FLAG_BAD_TOKEN | ssd.FLAG_BAD_HISTORY)
    assert mp.tolist() == [2, -1]
    assert nx[0].tolist() == [5, 4]
    assert nx[1].tolist() == [5, 7]


def test_backup_empty_and_argument_checks():
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    e = torch.empty(0, 3, dtype=torch.int32, device="cuda")
    ssd.ssd_ngram_backup(None, None, 0, 3, 10, torch.empty(0, 3, device="cuda"), e, status=z)
    with pytest.raises(ssd.SSDError):
        ssd.ssd_ngram_backup(None, None, 2, 3, 10, torch.zeros(1, 3, device="cuda"),
                             torch.zeros(1, 3, dtype=torch.int32, device="cuda"), status=z)
    with pytest.raises(ssd.SSDError):
        hist = torch.zeros(1, 8, dtype=torch.int32, device="cuda")
        ssd.ssd_ngram_backup(hist, z, 33, 3, 10, torch.zeros(1, 3, device="cuda"),
                             torch.zeros(1, 3, dtype=torch.int32, device="cuda"), status=z)
    # K = 0: only the match positions
    h = w.make_histories(w.tiny_histories(), seed=3)
    sp = h.spec
    mp = torch.full((sp.B,), -9, dtype=torch.int32, device="cuda")
    ssd.ssd_ngram_backup(dev(h.hist), dev(h.hist_len), sp.n, 0, sp.V,
                         torch.zeros(sp.B, 0, device="cuda"), None, slot=dev(h.slot),
                         match_pos=mp, status=z)
    _, rmp = oracle.ngram_backup(h.hist, h.hist_len, sp.n, 0, sp.V, h.slot,
                                 np.zeros((sp.B, 0), np.float32))
    np.testing.assert_array_equal(mp.cpu().numpy(), rmp)


# ---------------------------------------------------------------------------
# the batch plan
# ---------------------------------------------------------------------------
def gpu_plan(p, e, T_v, T_p, T_b, e_miss):
    nopt = len(T_b)
    o = {k: torch.full((nopt,), -1.0, dtype=torch.float64, device="cuda")
         for k in ("time", "tokens", "throughput", "speedup")}
    best = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ssd.ssd_fallback_plan(dev(np.asarray(p, np.float32)), dev(np.asarray(e, np.float32)), T_v, T_p,
                          T_b, e_miss, best=best, status=st, **o)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in o.items()}
    res["best"] = int(best.item())
    res["status"] = int(st.item())
    return res


def check_plan(p, e, T_v, T_p, T_b, e_miss):
    g = gpu_plan(p, e, T_v, T_p, T_b, e_miss)
    r = oracle.fallback_plan(np.asarray(p, np.float32), np.asarray(e, np.float32), T_v, T_p, T_b,
                             e_miss)
    for k in ("time", "tokens", "throughput", "speedup"):
        np.testing.assert_allclose(g[k], r[k], rtol=1e-12, atol=0)
    thr = r["throughput"]
    if np.sum(thr >= thr.max() * (1 - 1e-12)) == 1:
        assert g["best"] == r["best"]
    else:  # a near tie: any option within the rounding of the best is valid
        assert thr[g["best"]] >= thr.max() * (1 - 1e-12)
    return g


@pytest.mark.parametrize("B", [1, 7, 1000, 5000])
def test_plan_random(B):
    rng = np.random.default_rng(B)
    p = rng.uniform(0.6, 1.0, size=B)
    e = rng.uniform(1.0, 5.0, size=B)
    check_plan(p, e, 1.0, 0.45, [0.45, 0.05, 0.001], [2.2, 1.3, 1.0])


def test_plan_crossover_with_batch_size():
    best = []
    for B in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512):
        best.append(check_plan(np.full(B, 0.9), np.full(B, 3.0), 1.0, 0.5, [0.5, 0.02],
                               [2.8, 1.0])["best"])
    assert best[0] == 0 and best[-1] == 1


def test_plan_bad_rates_are_flagged_and_clamped():
    p = np.array([0.5, np.nan, 1.5, 0.9], np.float32)
    e = np.array([2.0, 3.0, -1.0, np.inf], np.float32)
    g = gpu_plan(p, e, 1.0, 0.5, [0.3], [1.0])
    assert g["status"] == ssd.FLAG_BAD_RATE
    r = oracle.fallback_plan(np.array([0.5, 0.0, 1.0, 0.9], np.float32),
                             np.array([2.0, 3.0, 0.0, 0.0], np.float32), 1.0, 0.5, [0.3], [1.0])
    np.testing.assert_allclose(g["time"], r["time"], rtol=1e-12)
    np.testing.assert_allclose(g["tokens"], r["tokens"], rtol=1e-12)


def test_plan_argument_checks():
    p = torch.ones(4, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for args in ((1.0, 0.5, [], []), (0.0, 0.0, [0.1], [1.0]), (1.0, -0.5, [0.1], [1.0]),
                 (1.0, 0.5, [float("nan")], [1.0]), (1.0, 0.5, [0.1] * 9, [1.0] * 9)):
        with pytest.raises(ssd.SSDError):
            ssd.ssd_fallback_plan(p, p, *args, status=st)
    with pytest.raises(ssd.SSDError):
        ssd.ssd_fallback_plan(p[:0], p[:0], 1.0, 0.5, [0.1], [1.0], status=st)


def test_policy_chain_on_device():
    """Plan from the hit rates, then the backup gated on the plan's choice,
    with no host round trip in between: at a large batch with a 90 % hit rate
    the random backup wins and the history is not searched."""
    h = w.make_histories(w.tiny_histories(), seed=3)
    sp = h.spec
    B = sp.B
    p = dev(np.full(B, 0.9, np.float32))
    e = dev(np.full(B, 3.0, np.float32))
    best = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ssd.ssd_fallback_plan(p, e, 1.0, 0.5, [0.5, 0.02], [2.8, 1.0], best=best, status=st)
    nxt = torch.full((B, sp.K), -7, dtype=torch.int32, device="cuda")
    mp = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    ssd.ssd_ngram_backup(dev(h.hist), dev(h.hist_len), sp.n, sp.K, sp.V, dev(h.u_rand), nxt,
                         slot=dev(h.slot), match_pos=mp, plan_best=best, random_option=1, status=st)
    torch.cuda.synchronize()
    assert int(best.item()) == 1 and int(st.item()) == 0
    rnx, rmp = oracle.ngram_backup(h.hist, h.hist_len, 0, sp.K, sp.V, h.slot, h.u_rand,
                                   next_tokens=np.full((B, sp.K), -7, np.int32))
    np.testing.assert_array_equal(nxt.cpu().numpy(), rnx)
    np.testing.assert_array_equal(mp.cpu().numpy(), rmp)

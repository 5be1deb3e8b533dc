"""GPU parity of tree-masked branch attention against the fp64 oracle
(outputs within 2e-2 absolute in bf16, log-sum-exp within 1e-3)."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_vocab_gb300 import binding as ssd
from speculative_decoding_vocab_gb300 import workloads as w

from parity import batched, gpu_attention, to_dev

pytestmark = pytest.mark.gpu
ATOL = 2e-2
LSE_ATOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_vocab_gb300 import build
    build.build()
    ssd.load()


def _check(ai, seqs=None, use_ws=True):
    out, lse, st = gpu_attention(ai, use_ws=use_ws)
    idx = np.arange(ai.spec.B) if seqs is None else np.asarray(seqs)
    ref, rlse, fl = batched(
        lambda q_, bt_, pl_, pa_: oracle.branch_attention(q_, ai.k_cache, ai.v_cache, bt_, pl_, pa_,
                                                          ai.spec.Hkv),
        len(idx), (ai.q[idx], ai.block_table[idx], ai.prefix_len[idx], ai.parent[idx]))
    err = np.abs(out[idx] - ref).max()
    lerr = np.abs(lse[idx] - rlse).max()
    assert err <= ATOL, f"max abs error {err}"
    assert lerr <= LSE_ATOL, f"lse max abs error {lerr}"
    assert st == 0
    return err


@pytest.mark.parametrize("spec", [
    w.AttnSpec(B=3, Hq=8, Hkv=2, d=64, L=100, tree="fanout", K=3, F=(3, 2, 1, 1), chain_len=4),
    w.AttnSpec(B=3, Hq=16, Hkv=1, d=128, L=77, tree="chain", n_chain=6, ragged_prefix=True),
    w.AttnSpec(B=2, Hq=4, Hkv=4, d=64, L=33, tree="fanout", K=4, F=(8, 4, 2, 1, 1), chain_len=4,
               ragged_chains=True, ragged_prefix=True),
    w.AttnSpec(B=2, Hq=8, Hkv=8, d=128, L=1, tree="fanout", K=2, F=(2, 1, 1), chain_len=2),
    w.AttnSpec(B=1, Hq=32, Hkv=2, d=64, L=0, tree="chain", n_chain=1),   # no prefix, one node
    w.AttnSpec(B=2, Hq=8, Hkv=1, d=128, L=500, tree="fanout", K=4, F=(20, 4, 2, 1, 1),
               chain_len=4),                                              # N = 116 nodes
    w.AttnSpec(B=2, Hq=16, Hkv=2, d=128, L=3000, tree="chain", n_chain=8,
               ragged_prefix=True),                     # 64 rows per KV head, keys split
], ids=["gqa4-d64", "gqa16-d128-chain", "ragged", "mha-d128", "single-node", "wide-tree",
        "d128-64rows-split"])
def test_small_shapes(spec):
    _check(w.make_attention(spec, seed=11))


@pytest.mark.parametrize("use_ws", [False, True], ids=["unsplit", "split"])
@pytest.mark.parametrize("spec", [
    w.AttnSpec(B=3, Hq=16, Hkv=1, d=128, L=77, tree="chain", n_chain=6, ragged_prefix=True),
    w.AttnSpec(B=2, Hq=16, Hkv=2, d=128, L=3000, tree="chain", n_chain=8, ragged_prefix=True),
    w.AttnSpec(B=2, Hq=8, Hkv=1, d=128, L=500, tree="fanout", K=4, F=(20, 4, 2, 1, 1), chain_len=4),
    w.AttnSpec(B=2, Hq=4, Hkv=2, d=64, L=200, tree="fanout", K=3, F=(3, 2, 1, 1), chain_len=4),
], ids=["d128-64rows", "d128-64rows-long", "d128-128rows", "d64"])
def test_without_lse(spec, use_ws):
    """A call without the log-sum-exp output (the d = 128 kernels then keep only
    the bf16 row sums): O bit-identical to the call with it, and within the
    tolerance of the oracle."""
    ai = w.make_attention(spec, seed=17)
    out_l, _, st_l = gpu_attention(ai, use_ws=use_ws)
    out_n, lse_n, st_n = gpu_attention(ai, use_ws=use_ws, want_lse=False)
    assert st_l == 0 and st_n == 0
    assert np.isnan(lse_n).all()  # nothing was written to the buffer that was not passed
    assert np.array_equal(out_n, out_l, equal_nan=True)
    ref, _, _ = oracle.branch_attention(ai.q, ai.k_cache, ai.v_cache, ai.block_table, ai.prefix_len,
                                        ai.parent, spec.Hkv)
    assert np.abs(out_n - ref).max() <= ATOL


@pytest.mark.parametrize("spec", [
    w.AttnSpec(B=2, Hq=4, Hkv=2, d=64, L=200, tree="chain", n_chain=128),
    w.AttnSpec(B=1, Hq=2, Hkv=1, d=128, L=90, tree="chain", n_chain=128, ragged_prefix=True),
], ids=["chain128-d64", "chain128-d128"])
def test_largest_trees(spec):
    """128 tree nodes, the most the attention call takes, all of them queries."""
    _check(w.make_attention(spec, seed=13))


def test_long_unsplit_keys_d128():
    """30,000 keys in one key range (no workspace): the block-table slice leaves
    no room for the six-stage d = 128 kernel, so the four-stage one runs."""
    spec = w.AttnSpec(B=1, Hq=8, Hkv=1, d=128, L=30000, tree="chain", n_chain=4)
    _check(w.make_attention(spec, seed=5), use_ws=False)


def test_draft_branch_attention_full():
    """The draft-shaped workload at full size: all 16 sequences."""
    ai = w.make_attention(w.draft_branch_attention(), seed=0)
    _check(ai)


def test_verify_attention_at_scale_full():
    """Full-size verify-shaped attention (B=64, L=8192, d=128): all 64 sequences."""
    spec = w.verify_attention_at_scale()
    ai = w.make_attention(spec, seed=0)
    _check(ai)


def test_flags_bad_tree_and_block():
    spec = w.AttnSpec(B=1, Hq=4, Hkv=2, d=64, L=40, tree="chain", n_chain=4)
    ai = w.make_attention(spec, seed=3)
    ai.parent[0, 2] = 3
    _, _, st = gpu_attention(ai)
    assert st & ssd.FLAG_BAD_TREE
    ai = w.make_attention(spec, seed=3)
    ai.block_table[0, 1] = 10 ** 6
    out, _, st = gpu_attention(ai)
    assert st & ssd.FLAG_BAD_BLOCK
    ref, _, _ = oracle.branch_attention(ai.q, ai.k_cache, ai.v_cache, ai.block_table, ai.prefix_len,
                                        ai.parent, spec.Hkv)
    assert np.abs(out - ref).max() <= ATOL


def test_flag_bad_prefix():
    """A prefix the block table cannot hold: the keys past it stay hidden (as in
    the oracle) and BAD_PREFIX is set; a negative prefix counts as 0."""
    spec = w.AttnSpec(B=2, Hq=8, Hkv=2, d=64, L=40, tree="chain", n_chain=4)
    ai = w.make_attention(spec, seed=4)
    maxb = ai.block_table.shape[1]
    ai.prefix_len[0] = 16 * maxb - 2
    ai.prefix_len[1] = -5
    out, lse, st = gpu_attention(ai)
    assert st & ssd.FLAG_BAD_PREFIX
    ref, rlse, fl = oracle.branch_attention(ai.q, ai.k_cache, ai.v_cache, ai.block_table,
                                            ai.prefix_len, ai.parent, spec.Hkv)
    assert np.all(fl & oracle.FLAG_BAD_PREFIX)
    assert np.abs(out - ref).max() <= ATOL
    assert np.abs(lse - rlse).max() <= LSE_ATOL


def test_attention_argument_errors():
    spec = w.AttnSpec(B=1, Hq=4, Hkv=2, d=64, L=40, tree="chain", n_chain=4)
    ai = w.make_attention(spec, seed=3)
    q = to_dev(ai.q)
    out = torch.empty_like(q)
    kc, vc = to_dev(ai.k_cache), to_dev(ai.v_cache)
    args = (to_dev(ai.block_table), to_dev(ai.prefix_len), to_dev(ai.parent))
    with pytest.raises(ssd.SSDError) as e:
        ssd.ssd_branch_attention(q[..., :32].contiguous(), kc[..., :32].contiguous(),
                                 vc[..., :32].contiguous(), *args, out[..., :32].contiguous())
    assert e.value.code == ssd.SSD_ERR_UNSUPPORTED
    with pytest.raises(ssd.SSDError) as e:
        ssd.ssd_branch_attention(q[:, :, :3].contiguous(), kc, vc, *args,
                                 out[:, :, :3].contiguous())
    assert e.value.code == ssd.SSD_ERR_INVALID_ARG

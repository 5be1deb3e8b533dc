"""CPU-side checks of the C ABI: the library builds and loads, exports every
call include/ssd.h declares, and its host-only logic (fan-out split, workspace
sizing, argument validation that returns before any launch) behaves as
documented.  No GPU work is issued here."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from speculative_decoding_vocab_gb300 import binding as ssd
from speculative_decoding_vocab_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssd.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ssd.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssd_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_calls():
    names = _declared()
    for n in ("ssd_verify", "ssd_predict_outcomes", "ssd_saguaro_sample", "ssd_cache_lookup",
              "ssd_branch_attention", "ssd_fanout_split", "ssd_workspace_size", "ssd_round"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in _declared():
        assert hasattr(lib, n), f"{n} declared in include/ssd.h but not exported"
    for n in ssd.EXPORTS:
        assert n in _declared()


def test_status_strings(lib):
    for code in range(5):
        assert lib.ssd_status_string(code)


@pytest.mark.parametrize("budget,K,r", [(9, 4, 0.5), (32, 5, 0.5), (64, 4, 0.5), (16, 4, 0.5),
                                        (100, 7, 0.3), (17, 16, 0.9), (5, 0, 0.5), (1000, 3, 1.0)])
def test_fanout_split_matches_oracle(lib, budget, K, r):
    assert ssd.ssd_fanout_split(budget, K, r) == oracle.fanout_split(budget, K, r)


def test_fanout_split_errors(lib):
    F = (ctypes.c_int32 * 8)()
    assert lib.ssd_fanout_split(3, 4, 0.5, F) == ssd.SSD_ERR_INVALID_ARG
    assert lib.ssd_fanout_split(9, 4, 0.0, F) == ssd.SSD_ERR_INVALID_ARG
    assert lib.ssd_fanout_split(9, 4, 1.5, F) == ssd.SSD_ERR_INVALID_ARG
    assert lib.ssd_fanout_split(9, 4, 0.5, None) == ssd.SSD_ERR_INVALID_ARG


def test_workspace_size(lib):
    F = (16, 8, 4, 2, 1, 1)
    n = ssd.ssd_workspace_size(32, 5, 128256, "bf16", F)
    assert n > 0 and n % 256 == 0
    assert ssd.ssd_workspace_size(64, 5, 128256, "bf16", F) > n
    assert ssd.ssd_workspace_size(32, 5, 8, "bf16", (16, 8, 4, 2, 1, 1)) == 0  # F_k > V
    assert ssd.ssd_workspace_size(2, 17, 1000, "f32", tuple([1] * 18)) == 0   # K > 16
    assert ssd.ssd_workspace_size(2, 1, 1000, "f32", (300, 1)) == 0          # F > 256
    # rows up to 4 MiB: V = 2^21 in bf16, 2^20 in fp32; one element more is unsupported
    assert ssd.ssd_workspace_size(2, 2, 1 << 21, "bf16", (16, 4, 1)) > 0
    assert ssd.ssd_workspace_size(2, 2, (1 << 21) + 8, "bf16", (16, 4, 1)) == 0
    assert ssd.ssd_workspace_size(2, 2, 1 << 20, "f32", (16, 4, 1)) > 0
    assert ssd.ssd_workspace_size(2, 2, (1 << 20) + 4, "f32", (16, 4, 1)) == 0


def test_attention_workspace_size(lib):
    """Key-split partials: O (d floats) and (m, l, unrounded l) per row of every
    split, in two 256-byte aligned arrays; none when the work items already fill
    the GPU."""
    B, Hkv, d = 64, 8, 128
    per_split = B * Hkv * 128 * d * 4 + B * Hkv * 128 * 3 * 4  # one row tile per KV head
    n = ssd.ssd_attention_workspace_size(B, 6, 64, Hkv, d, 8192)
    assert n > 0 and n % per_split == 0 and 2 <= n // per_split <= 16
    # draft tree shape: its 256 row tiles run as pipelines without splitting the keys
    assert ssd.ssd_attention_workspace_size(16, 64, 32, 8, 64, 2048) == 0
    assert ssd.ssd_attention_workspace_size(2, 6, 12, 8, 128, 100) == 0    # Hq % Hkv != 0
    assert ssd.ssd_attention_workspace_size(0, 6, 64, 8, 128, 100) == 0    # no sequences


def _F(F):
    return (ctypes.c_int32 * len(F))(*F)


def test_validation_returns_before_any_launch(lib):
    """Fake device addresses: every call below must fail its host checks."""
    F = _F((2, 1, 1))
    good = ctypes.c_void_p(0x100000)
    odd = ctypes.c_void_p(0x100004)
    ws_n = lib.ssd_workspace_size(2, 2, 1000, ssd.SSD_F32, F)
    # misaligned logits
    assert lib.ssd_saguaro_sample(odd, ssd.SSD_F32, 3000, 1000, 2, 2, 1000, F, 0.5, 1.0, good, good,
                                  None, good, good, ws_n, None) == ssd.SSD_ERR_UNSUPPORTED
    # row stride not a multiple of 16 bytes
    assert lib.ssd_saguaro_sample(good, ssd.SSD_F32, 3003, 1001, 2, 2, 1000, F, 0.5, 1.0, good, good,
                                  None, good, good, ws_n, None) == ssd.SSD_ERR_UNSUPPORTED
    # C out of range, negative temperature
    assert lib.ssd_saguaro_sample(good, ssd.SSD_F32, 3000, 1000, 2, 2, 1000, F, 1.5, 1.0, good, good,
                                  None, good, good, ws_n, None) == ssd.SSD_ERR_INVALID_ARG
    assert lib.ssd_saguaro_sample(good, ssd.SSD_F32, 3000, 1000, 2, 2, 1000, F, 0.5, -1.0, good,
                                  good, None, good, good, ws_n, None) == ssd.SSD_ERR_INVALID_ARG
    # workspace too small or missing
    assert lib.ssd_verify(good, good, ssd.SSD_F32, 3000, 1000, 2, 2, 1000, F, 0.5, 1.0, good, good,
                          good, good, good, good, None, None, None, good, good, ws_n - 256,
                          None) == ssd.SSD_ERR_WORKSPACE
    assert lib.ssd_round(good, good, ssd.SSD_F32, 3000, 1000, 2, 2, 1000, F, 0.5, 1.0, good, good,
                         good, None, good, None, good, good, good, None, None, None, None, None,
                         None, None, None, good, None, 0, None) == ssd.SSD_ERR_WORKSPACE
    # the no-allocation entry point maps argument errors as ssd_verify does,
    # before its scratch-size check
    assert lib.ssd_verify_noalloc(good, good, ssd.SSD_F32, 3000, 1000, 2, 2, 1000, _F((-1, 1, 1)),
                                  0.5, 1.0, good, good, good, good, good, good, None, None, None,
                                  good, None) == ssd.SSD_ERR_INVALID_ARG
    assert lib.ssd_verify_noalloc(good, good, 7, 3000, 1000, 2, 2, 1000, F, 0.5, 1.0, good, good,
                                  good, good, good, good, None, None, None, good,
                                  None) == ssd.SSD_ERR_INVALID_ARG
    assert lib.ssd_verify_noalloc(good, good, ssd.SSD_F32, 3000, 1000, 2, 2, 1000, F, 1.5, 1.0, good,
                                  good, good, good, good, good, None, None, None, good,
                                  None) == ssd.SSD_ERR_INVALID_ARG
    assert lib.ssd_verify_noalloc(odd, good, ssd.SSD_F32, 3000, 1000, 2, 2, 1000, F, 0.5, 1.0, good,
                                  good, good, good, good, good, None, None, None, good,
                                  None) == ssd.SSD_ERR_UNSUPPORTED
    # F_k > V
    assert lib.ssd_predict_outcomes(good, ssd.SSD_BF16, 3008, 1008, 2, 2, 4, _F((8, 1, 1)), 1.0,
                                    good, None, good, good, 1 << 20, None) == ssd.SSD_ERR_UNSUPPORTED
    # lookup: K out of range
    assert lib.ssd_cache_lookup(good, None, 2, 17, _F(tuple([1] * 18)), good, good, good, None, None,
                                good, None) == ssd.SSD_ERR_INVALID_ARG
    # attention: head dim, GQA ratio, tree size
    args = [good, good, good, good, 4, 100, good, good]
    assert lib.ssd_branch_attention(*args, 2, 4, 4, 8, 2, 96, 0.1, good, None, good, None, 0,
                                    None) == ssd.SSD_ERR_UNSUPPORTED
    assert lib.ssd_branch_attention(*args, 2, 4, 4, 6, 4, 64, 0.1, good, None, good, None, 0,
                                    None) == ssd.SSD_ERR_INVALID_ARG
    assert lib.ssd_branch_attention(*args, 2, 200, 4, 8, 2, 64, 0.1, good, None, good, None, 0,
                                    None) == ssd.SSD_ERR_UNSUPPORTED
    assert lib.ssd_branch_attention(*args, 2, 4, 5, 8, 2, 64, 0.1, good, None, good, None, 0,
                                    None) == ssd.SSD_ERR_UNSUPPORTED


def test_binding_refuses_host_tensors(lib):
    import torch
    with pytest.raises(ValueError, match="CUDA device"):
        ssd._ptr(torch.zeros(4))


def test_binding_refuses_other_layouts_and_dtypes():
    """The library reads arrays as dense row-major memory of the header's C
    type: a column-major gather (numpy's a[:, idx]) or a float64 uniform
    array is refused before any pointer is taken."""
    import torch
    a = np.arange(12, dtype=np.int32).reshape(3, 4)[:, np.array([0, 2, 1])]
    assert not a.flags["C_CONTIGUOUS"]
    with pytest.raises(ValueError, match="contiguous"):
        ssd._ptr(torch.from_numpy(a), torch.int32)
    with pytest.raises(ValueError, match="float32"):
        ssd._ptr(torch.zeros(4, dtype=torch.float64), torch.float32)
    # strided logits pass the layout check (their strides go to the call)
    with pytest.raises(ValueError, match="CUDA device"):
        ssd._ptr(torch.zeros(4, 8)[:, :5], strided=True)
    # the numpy helper makes any layout dense
    assert ssd.tensor(a, "cpu").is_contiguous()


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        ssd.load(str(tmp_path / "nope.so"))


def test_fallback_fill_tree_argument_checks(lib):
    """Host validation of the miss-fallback, cache-fill and tree calls: every
    case here is refused (or is an empty batch) before any launch."""
    E = ssd
    nul = None
    fake = ctypes.c_void_p(16)  # never dereferenced: each call returns before a launch
    # n-gram backup: n or K out of range, negative sizes, empty batch
    assert lib.ssd_ngram_backup(fake, 8, fake, 1, 33, 4, 10, nul, fake, nul, 0, fake, nul, fake, nul) == E.SSD_ERR_UNSUPPORTED
    assert lib.ssd_ngram_backup(fake, 8, fake, 1, 3, 1025, 10, nul, fake, nul, 0, fake, nul, fake, nul) == E.SSD_ERR_UNSUPPORTED
    assert lib.ssd_ngram_backup(fake, 8, fake, -1, 3, 4, 10, nul, fake, nul, 0, fake, nul, fake, nul) == E.SSD_ERR_INVALID_ARG
    assert lib.ssd_ngram_backup(fake, 8, fake, 1, 3, 4, 0, nul, fake, nul, 0, fake, nul, fake, nul) == E.SSD_ERR_INVALID_ARG
    assert lib.ssd_ngram_backup(nul, 8, nul, 1, 3, 4, 10, nul, fake, nul, 0, fake, nul, fake, nul) == E.SSD_ERR_INVALID_ARG
    assert lib.ssd_ngram_backup(nul, 0, nul, 0, 3, 4, 10, nul, nul, nul, 0, nul, nul, nul, nul) == E.SSD_OK
    # plan: empty batch, too many options, bad timings
    tb = (ctypes.c_double * 9)(*([0.1] * 9))
    em = (ctypes.c_double * 9)(*([1.0] * 9))
    assert lib.ssd_fallback_plan(fake, fake, 0, 1.0, 0.5, 1, tb, em, nul, nul, nul, nul, nul, fake, nul) == E.SSD_ERR_INVALID_ARG
    assert lib.ssd_fallback_plan(fake, fake, 4, 1.0, 0.5, 9, tb, em, nul, nul, nul, nul, nul, fake, nul) == E.SSD_ERR_UNSUPPORTED
    assert lib.ssd_fallback_plan(fake, fake, 4, 0.0, 0.0, 1, tb, em, nul, nul, nul, nul, nul, fake, nul) == E.SSD_ERR_INVALID_ARG
    assert lib.ssd_fallback_plan(fake, fake, 4, 1.0, -1.0, 1, tb, em, nul, nul, nul, nul, nul, fake, nul) == E.SSD_ERR_INVALID_ARG
    # K/V append: d not a multiple of 8 or above 256, empty batch
    assert lib.ssd_kv_append(fake, fake, fake, fake, fake, 4, 8, fake, 0, 2, 3, 2, 12, fake, nul) == E.SSD_ERR_UNSUPPORTED
    assert lib.ssd_kv_append(fake, fake, fake, fake, fake, 4, 8, fake, 0, 2, 3, 2, 264, fake, nul) == E.SSD_ERR_UNSUPPORTED
    assert lib.ssd_kv_append(fake, fake, fake, fake, fake, 0, 8, fake, 0, 2, 3, 2, 64, fake, nul) == E.SSD_ERR_INVALID_ARG
    assert lib.ssd_kv_append(nul, nul, nul, nul, nul, 4, 8, nul, 0, 0, 3, 2, 64, nul, nul) == E.SSD_OK
    # per-branch draw: column past the payload, C outside (0, 1], workspace missing
    assert lib.ssd_fill_sample(fake, E.SSD_F32, 16, 1, 2, 16, 2, 0.5, 1.0, fake, 3, 3, fake, nul, fake, fake, nul, 0, nul) == E.SSD_ERR_INVALID_ARG
    assert lib.ssd_fill_sample(fake, E.SSD_F32, 16, 1, 2, 16, 2, 0.0, 1.0, fake, 0, 3, fake, nul, fake, fake, nul, 1 << 20, nul) == E.SSD_ERR_INVALID_ARG
    assert lib.ssd_fill_sample(fake, E.SSD_F32, 16, 1, 2, 16, 2, 0.5, 1.0, fake, 0, 3, fake, nul, fake, fake, nul, 0, nul) == E.SSD_ERR_WORKSPACE
    # tree: too many nodes, rows above 512 KiB, bad temperature, empty batch
    assert lib.ssd_tree_verify(fake, fake, E.SSD_F32, 0, 16, 1, 257, 16, 1.0, fake, fake, fake, fake, fake, fake, fake, nul, nul, fake, nul) == E.SSD_ERR_UNSUPPORTED
    assert lib.ssd_tree_verify(fake, fake, E.SSD_F32, 0, 131080, 1, 2, 131080, 1.0, fake, fake, fake, fake, fake, fake, fake, nul, nul, fake, nul) == E.SSD_ERR_UNSUPPORTED
    assert lib.ssd_tree_verify(fake, fake, E.SSD_F32, 0, 16, 1, 2, 16, -1.0, fake, fake, fake, fake, fake, fake, fake, nul, nul, fake, nul) == E.SSD_ERR_INVALID_ARG
    assert lib.ssd_tree_verify(nul, nul, E.SSD_BF16, 0, 16, 0, 2, 16, 1.0, nul, nul, nul, nul, nul, nul, nul, nul, nul, nul, nul) == E.SSD_OK

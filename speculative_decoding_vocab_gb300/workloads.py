"""Seeded synthetic inputs for one speculation round and for branch attention.

This module is input plumbing only: it draws random numbers and shapes them
into the tensors a round consumes.  It holds none of the method's arithmetic
(no softmax, no acceptance test, no sampling rule, no attention), so both the
CUDA path and the fp64 oracle can read the very same bytes from it.

Contents
--------
* ``philox4x32_10`` -- the counter-based generator of Salmon, Moraes, Dror and
  Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11), written from
  that paper's definition (Philox-4x32 with 10 rounds).  Every uniform a round
  consumes (draft draws, acceptance draws, bonus draws) comes from it, keyed by
  the seed and counted by (round, sequence, slot kind, slot index).
* logit generators for the two workload shapes the speculative-speculative
  decoding pages evaluate on (Llama-3 and Qwen-3 vocabularies): i.i.d.
  Gaussian logits and Zipf-shaped logits over a seeded permutation, with the
  draft equal to the target plus Gaussian noise.
* paged KV caches, block tables and branch trees for tree-masked attention.
* branch-decode (cache fill) steps: per step the draft logits of every
  branch, the key/value rows of the fed tokens and the step-major branch tree.
* token trees for multi-candidate verification: a level-order tree of given
  branching and per-node target / draft logit rows (the children's tokens
  are drawn by the caller from the draft rows).
* token histories for the miss fallback: Zipf-distributed tokens in which
  spans repeat earlier spans (the repetition an n-gram backup feeds on), with
  a seeded set of sequences that missed the speculation cache.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# ---------------------------------------------------------------------------
# Philox4x32-10 (Salmon et al., SC'11, section 4 "Philox")
# ---------------------------------------------------------------------------
_PHILOX_M0 = np.uint64(0xD2511F53)
_PHILOX_M1 = np.uint64(0xCD9E8D57)
_PHILOX_W0 = np.uint32(0x9E3779B9)  # golden ratio
_PHILOX_W1 = np.uint32(0xBB67AE85)  # sqrt(3) - 1
_MASK32 = np.uint64(0xFFFFFFFF)

# slot kinds of the counter's third word
SLOT_DRAFT = 0   # u_draft[b, j]: the uniform the draft's inverse-CDF draw uses
SLOT_ACCEPT = 1  # u_acc[b, j]: the uniform of the acceptance test at position j
SLOT_BONUS = 2   # u_bonus[b]: the uniform of the residual / bonus draw
SLOT_BACKUP = 3  # u_rand[b, t]: the uniform of the random-token backup at position t
SLOT_FILL = 4    # u_fill[b, t*S + s]: the uniform of branch s's draw at decode step t
SLOT_TREE = 5    # u_acc[b, m]: the uniform of tree node m's acceptance test
SLOT_TREE_BONUS = 6  # u_bonus[b]: the uniform of the tree walk's bonus draw


def philox4x32_10(counter: np.ndarray, key: tuple[int, int]) -> np.ndarray:
    """Philox-4x32 with 10 rounds on a batch of 128-bit counters.

    ``counter`` is ``uint32[..., 4]``; ``key`` is two 32-bit words.  Each round
    multiplies words 0 and 2 by the two Philox multipliers, splits the 64-bit
    products into high and low halves, and mixes the high halves with words 1
    and 3 and the round key; the key is bumped by the two Weyl constants
    between rounds.  Returns ``uint32[..., 4]``.
    """
    c = np.asarray(counter, dtype=np.uint32)
    c0 = c[..., 0].astype(np.uint64)
    c1 = c[..., 1].astype(np.uint64)
    c2 = c[..., 2].astype(np.uint64)
    c3 = c[..., 3].astype(np.uint64)
    k0 = np.uint32(key[0] & 0xFFFFFFFF)
    k1 = np.uint32(key[1] & 0xFFFFFFFF)
    for rnd in range(10):
        if rnd:
            k0 = np.uint32((int(k0) + int(_PHILOX_W0)) & 0xFFFFFFFF)
            k1 = np.uint32((int(k1) + int(_PHILOX_W1)) & 0xFFFFFFFF)
        prod0 = _PHILOX_M0 * c0
        prod1 = _PHILOX_M1 * c2
        hi0, lo0 = prod0 >> np.uint64(32), prod0 & _MASK32
        hi1, lo1 = prod1 >> np.uint64(32), prod1 & _MASK32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint64(k0),
                          lo1,
                          hi0 ^ c3 ^ np.uint64(k1),
                          lo0)
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def uniforms_from_bits(x: np.ndarray) -> np.ndarray:
    """Map 32 random bits to a uniform in [0, 1) with 24 significant bits.

    u = (x >> 8) * 2^-24 is exact in both float32 and float64, so the GPU and
    the oracle see the identical number.
    """
    return ((np.asarray(x, dtype=np.uint32) >> np.uint32(8)).astype(np.float64)
            * 2.0 ** -24).astype(np.float32)


def round_uniforms(seed: int, rnd: int, B: int, K: int):
    """The three uniform arrays of one round: ``u_draft[B,K]``, ``u_acc[B,K]``, ``u_bonus[B]``.

    Counter = (round, sequence, slot kind, slot index); key = (seed low, seed high).
    """
    key = (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)

    def draw(kind, n):
        b = np.arange(B, dtype=np.uint32)[:, None]
        j = np.arange(n, dtype=np.uint32)[None, :]
        ctr = np.stack(np.broadcast_arrays(np.uint32(rnd & 0xFFFFFFFF), b,
                                           np.uint32(kind), j), axis=-1)
        return uniforms_from_bits(philox4x32_10(ctr, key)[..., 0])

    return draw(SLOT_DRAFT, K), draw(SLOT_ACCEPT, K), draw(SLOT_BONUS, 1)[:, 0].copy()


# ---------------------------------------------------------------------------
# bf16 helpers (bit-level, round-to-nearest-even)
# ---------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite float32 to bfloat16 (nearest, ties to even); returns the uint16 bits.

    +-inf map to +-inf; NaN inputs are not supported.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    inf = (b & np.uint32(0x7FFFFFFF)) == np.uint32(0x7F800000)
    rounded = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    out = rounded.astype(np.uint16)
    if inf.any():
        out[inf] = (b[inf] >> np.uint32(16)).astype(np.uint16)
    return out


def _bf16_normals(rng, shape, chunk=1 << 24) -> np.ndarray:
    """bf16 bits of N(0, 1) draws, generated in bounded chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    for o in range(0, n, chunk):
        m = min(chunk, n - o)
        out[o:o + m] = f32_to_bf16_bits(rng.standard_normal(m, dtype=np.float32))
    return out.reshape(shape)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------------------
# Round-step workloads
# ---------------------------------------------------------------------------
@dataclass
class RoundSpec:
    """Shape and value recipe of one batched speculation round."""
    B: int
    K: int
    V: int
    dtype: str                 # "f32" or "bf16"
    recipe: str                # "gauss" or "zipf"
    T: float = 1.0
    C: float = 1.0
    budget: int = 0
    F: tuple = ()              # fan-out (F_0..F_K); filled from the budget when empty
    target_sigma: float = 2.0  # gauss recipe: target logits ~ N(0, sigma^2)
    zipf_slope: float = 1.1    # zipf recipe: -slope * ln(rank)
    target_noise: float = 0.3  # zipf recipe: N(0, noise^2) added to the target
    draft_noise: float = 0.5   # draft = target + N(0, draft_noise^2)
    row_pad: int = 0           # extra elements at the end of every row (ragged strides)
    name: str = ""


@dataclass
class RoundInputs:
    spec: RoundSpec
    target: np.ndarray         # [B, K+1, V + row_pad] float32 or uint16 (bf16 bits)
    draft: np.ndarray          # same
    u_draft: np.ndarray        # [B, K] float32
    u_acc: np.ndarray          # [B, K] float32
    u_bonus: np.ndarray        # [B] float32
    payload: np.ndarray = field(default=None)  # [B, sumF, K] int32 cache contents

    @property
    def row_stride(self) -> int:
        return self.target.shape[-1]


def _gauss_rows(rng, rows, V, sigma_t, sigma_d):
    zt = rng.standard_normal((rows, V), dtype=np.float32) * np.float32(sigma_t)
    zd = zt + rng.standard_normal((rows, V), dtype=np.float32) * np.float32(sigma_d)
    return zt, zd


def _zipf_rows(rng, rows, V, slope, noise_t, noise_d):
    base = (-slope * np.log(np.arange(1, V + 1, dtype=np.float64))).astype(np.float32)
    perm = rng.permuted(np.broadcast_to(np.arange(V, dtype=np.int32), (rows, V)), axis=1)
    zt = base[perm] + rng.standard_normal((rows, V), dtype=np.float32) * np.float32(noise_t)
    zd = zt + rng.standard_normal((rows, V), dtype=np.float32) * np.float32(noise_d)
    return zt, zd


def make_round(spec: RoundSpec, seed: int = 0, rnd: int = 0, payload: bool = True) -> RoundInputs:
    """Seeded logits, uniforms and cache payload of round ``rnd``.

    Rows are generated per sequence from a generator keyed by (seed, round,
    sequence), so a sample of sequences can be regenerated on its own.
    """
    B, K, V = spec.B, spec.K, spec.V
    W = V + spec.row_pad
    if spec.dtype == "f32":
        target = np.zeros((B, K + 1, W), np.float32)
        draft = np.zeros((B, K + 1, W), np.float32)
    else:
        target = np.zeros((B, K + 1, W), np.uint16)
        draft = np.zeros((B, K + 1, W), np.uint16)
    for b in range(B):
        zt, zd = sequence_logits(spec, seed, rnd, b)
        if spec.dtype == "f32":
            target[b, :, :V] = zt
            draft[b, :, :V] = zd
        else:
            target[b, :, :V] = f32_to_bf16_bits(zt)
            draft[b, :, :V] = f32_to_bf16_bits(zd)
    u_draft, u_acc, u_bonus = round_uniforms(seed, rnd, B, K)
    pl = None
    if payload:
        sumF = int(sum(spec.F))
        rng = np.random.default_rng(np.random.SeedSequence([seed, rnd, 0x5107]))
        pl = rng.integers(0, V, size=(B, sumF, K), dtype=np.int32)
    return RoundInputs(spec, target, draft, u_draft, u_acc, u_bonus, pl)


def sequence_logits(spec: RoundSpec, seed: int, rnd: int, b: int):
    """float32 target and draft logits ``[K+1, V]`` of sequence ``b`` (before bf16 rounding)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, rnd, b, 0x10617]))
    if spec.recipe == "gauss":
        return _gauss_rows(rng, spec.K + 1, spec.V, spec.target_sigma, spec.draft_noise)
    if spec.recipe == "zipf":
        return _zipf_rows(rng, spec.K + 1, spec.V, spec.zipf_slope, spec.target_noise,
                          spec.draft_noise)
    raise ValueError(f"unknown recipe {spec.recipe!r}")


# The five workloads: the tiny Gaussian round, the Llama-3 vocabulary round, the
# large-batch Qwen-3 vocabulary round, draft-shaped branch attention and
# verify-shaped attention at scale (plus its round).
def tiny_round() -> RoundSpec:
    return RoundSpec(B=1, K=4, V=4096, dtype="f32", recipe="gauss", T=1.0, C=0.5,
                     F=(4, 2, 1, 1, 1), budget=9, target_sigma=2.0, draft_noise=0.5,
                     name="tiny-gauss-B1-K4-V4096-f32")


def llama3_round(T: float = 1.0, B: int = 32) -> RoundSpec:
    return RoundSpec(B=B, K=5, V=128256, dtype="bf16", recipe="zipf", T=T, C=1.0,
                     budget=32, F=(16, 8, 4, 2, 1, 1), draft_noise=1.0,
                     name=f"llama3-vocab-B{B}-K5-V128256-bf16-T{T:g}")


def qwen3_round(C: float = 1.0, B: int = 256) -> RoundSpec:
    return RoundSpec(B=B, K=4, V=151936, dtype="bf16", recipe="zipf", T=0.6, C=C,
                     budget=64, F=(33, 17, 8, 4, 2), draft_noise=1.5,
                     name=f"qwen3-vocab-B{B}-K4-V151936-bf16-C{C:g}")


def llama3_round_at_scale(B: int = 64) -> RoundSpec:
    return RoundSpec(B=B, K=5, V=128256, dtype="bf16", recipe="zipf", T=1.0, C=1.0,
                     budget=32, F=(16, 8, 4, 2, 1, 1), draft_noise=1.0,
                     name=f"llama3-vocab-B{B}-K5-V128256-bf16-scale")


# ---------------------------------------------------------------------------
# Branch-attention workloads
# ---------------------------------------------------------------------------
PAGE = 16  # tokens per KV-cache block


def branch_tree(K: int, F, chain_lens) -> np.ndarray:
    """Parent indices of the speculation tree of one sequence.

    Nodes 0..K-1 are the spine (the K draft tokens, a chain hanging off the
    prefix); then, for each depth a = 0..K, F_a chains (a guessed bonus token
    followed by its pre-speculated continuation) hang off spine node a-1, or off
    the prefix end when a = 0.  ``chain_lens`` gives the length of every chain in
    that order.  -1 marks the prefix end.
    """
    parent = [-1 if m == 0 else m - 1 for m in range(K)]
    c = 0
    for a in range(K + 1):
        for _ in range(F[a]):
            n = int(chain_lens[c])
            c += 1
            first = len(parent)
            for t in range(n):
                parent.append((a - 1) if t == 0 else first + t - 1)
    return np.asarray(parent, dtype=np.int32)


def chain_tree(n: int) -> np.ndarray:
    """A plain chain of n nodes (causal rows after the prefix)."""
    return np.asarray([-1] + list(range(n - 1)), dtype=np.int32)[:n]


@dataclass
class AttnSpec:
    B: int
    Hq: int
    Hkv: int
    d: int
    L: int                     # prefix length (maximum when ragged)
    tree: str                  # "fanout" or "chain"
    K: int = 4
    F: tuple = (8, 4, 2, 1, 1)
    chain_len: int = 4
    n_chain: int = 6           # chain tree length
    ragged_prefix: bool = False
    ragged_chains: bool = False
    name: str = ""


@dataclass
class AttnInputs:
    spec: AttnSpec
    q: np.ndarray              # [B, Nq, Hq, d] uint16 (bf16 bits)
    k_cache: np.ndarray        # [nb, Hkv, PAGE, d] uint16
    v_cache: np.ndarray        # [nb, Hkv, PAGE, d] uint16
    block_table: np.ndarray    # [B, maxb] int32 (-1 past the end)
    prefix_len: np.ndarray     # [B] int32
    parent: np.ndarray         # [B, N] int32
    N: int
    Nq: int


def draft_branch_attention(B: int = 16) -> AttnSpec:
    return AttnSpec(B=B, Hq=32, Hkv=8, d=64, L=2048, tree="fanout", K=4, F=(8, 4, 2, 1, 1),
                    chain_len=4, name=f"branch-attn-draft-B{B}-Hq32-Hkv8-d64-L2048-N68")


def verify_attention_at_scale(B: int = 64) -> AttnSpec:
    return AttnSpec(B=B, Hq=64, Hkv=8, d=128, L=8192, tree="chain", n_chain=6,
                    name=f"verify-attn-B{B}-Hq64-Hkv8-d128-L8192-N6")


def attn_tree(spec: AttnSpec, rng) -> np.ndarray:
    if spec.tree == "chain":
        return chain_tree(spec.n_chain)
    nchains = int(sum(spec.F))
    if spec.ragged_chains:
        lens = rng.integers(1, spec.chain_len + 1, size=nchains)
    else:
        lens = np.full(nchains, spec.chain_len)
    return branch_tree(spec.K, spec.F, lens)


def make_attention(spec: AttnSpec, seed: int = 0, values: str = "normal") -> AttnInputs:
    """Seeded Q, paged K/V caches, block table, prefix lengths and tree.

    Every sequence gets the same tree shape (ragged chains draw one shape for
    the batch); its K/V rows for logical positions 0 .. L_b + N - 1 live in
    blocks picked by a seeded permutation of the physical block pool.
    """
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0xA77E]))
    parent1 = attn_tree(spec, rng)
    N = int(parent1.shape[0])
    Nq = N - spec.K if spec.tree == "fanout" else N
    B = spec.B
    if spec.ragged_prefix:
        prefix = rng.integers(1, spec.L + 1, size=B).astype(np.int32)
    else:
        prefix = np.full(B, spec.L, np.int32)
    nblk = [(int(prefix[b]) + N + PAGE - 1) // PAGE for b in range(B)]
    nb = int(sum(nblk))
    maxb = max(nblk)
    phys = rng.permutation(nb).astype(np.int32)
    table = np.full((B, maxb), -1, np.int32)
    o = 0
    for b in range(B):
        table[b, :nblk[b]] = phys[o:o + nblk[b]]
        o += nblk[b]
    shape_kv = (nb, spec.Hkv, PAGE, spec.d)
    if values == "normal":
        q = _bf16_normals(rng, (B, Nq, spec.Hq, spec.d))
        kc = _bf16_normals(rng, shape_kv)
        vc = _bf16_normals(rng, shape_kv)
    else:
        raise ValueError(values)
    parent = np.broadcast_to(parent1, (B, N)).copy()
    return AttnInputs(spec, q, kc, vc, table, prefix, parent, N, Nq)


def attention_bytes(spec: AttnSpec, N: int, Nq: int, prefix_len) -> int:
    """Algorithmic HBM bytes of one call: every visible K/V row read once per
    (sequence, KV head), plus Q read and O written once (bf16)."""
    kv = sum(2 * (int(L) + N) * spec.Hkv * spec.d * 2 for L in prefix_len)
    qo = 2 * spec.B * Nq * spec.Hq * spec.d * 2
    return kv + qo


def round_bytes(spec: RoundSpec) -> int:
    """Algorithmic HBM bytes of one verify+predict round: every target and draft
    logit read once."""
    elem = 4 if spec.dtype == "f32" else 2
    return 2 * spec.B * (spec.K + 1) * spec.V * elem


# ---------------------------------------------------------------------------
# Cache fill by branch decode
# ---------------------------------------------------------------------------
@dataclass
class FillSpec:
    """Shape and value recipe of a speculation-cache fill: K decode steps over
    the S = sum(F) branches of B sequences, with tree attention of shape
    (Hq, Hkv, d) over a prefix of L tokens."""
    B: int
    K: int
    F: tuple
    V: int
    dtype: str
    T: float
    C: float
    Hq: int
    Hkv: int
    d: int
    L: int
    recipe: str = "zipf"       # draft logits: "zipf" (slope 1.1 + N(0,1)) or "gauss" (N(0, 2^2))
    name: str = ""

    @property
    def S(self) -> int:
        return int(sum(self.F))


def fill_tree(K: int, F, steps: int) -> np.ndarray:
    """Parent indices after ``steps`` decode steps, numbered step-major: nodes
    0..K-1 are the spine (the round's draft tokens); node K + t*S + s is the
    token branch s fed at step t.  Step 0 feeds each branch's guessed bonus,
    hung off spine node a-1 for a slot of depth a (the prefix end for a = 0);
    step t > 0 feeds the token drawn at step t-1, hung off the branch's
    previous node.  The nodes fed at a step are the last S nodes."""
    S = int(sum(F))
    depth = np.repeat(np.arange(K + 1), F)
    parent = [-1 if m == 0 else m - 1 for m in range(K)]
    for t in range(steps):
        for s in range(S):
            parent.append(int(depth[s]) - 1 if t == 0 else K + (t - 1) * S + s)
    return np.asarray(parent, dtype=np.int32)


def fill_uniforms(seed: int, rnd: int, t: int, B: int, S: int) -> np.ndarray:
    """``u[B, S]`` of decode step ``t`` (Philox counter (round, sequence,
    SLOT_FILL, t*S + s))."""
    key = (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    b = np.arange(B, dtype=np.uint32)[:, None]
    j = (t * S + np.arange(S, dtype=np.uint32))[None, :]
    ctr = np.stack(np.broadcast_arrays(np.uint32(rnd & 0xFFFFFFFF), b, np.uint32(SLOT_FILL),
                                       j.astype(np.uint32)), axis=-1)
    return uniforms_from_bits(philox4x32_10(ctr, key)[..., 0])


def fill_step_logits(spec: FillSpec, seed: int, t: int, seqs=None) -> np.ndarray:
    """Draft logits [len(seqs), S, V] of step ``t`` (float32, or bf16 bits),
    generated per (seed, step, sequence)."""
    seqs = range(spec.B) if seqs is None else seqs
    out = []
    for b in seqs:
        rng = np.random.default_rng(np.random.SeedSequence([seed, t, b, 0xF111]))
        if spec.recipe == "zipf":
            _, zd = _zipf_rows(rng, spec.S, spec.V, 1.1, 0.0, 1.0)
        else:
            zd = rng.standard_normal((spec.S, spec.V), dtype=np.float32) * np.float32(2.0)
        out.append(zd if spec.dtype == "f32" else f32_to_bf16_bits(zd))
    return np.stack(out)


def fill_step_kv(spec: FillSpec, seed: int, t: int):
    """bf16 bits of the key and value rows [B, S, Hkv, d] of the tokens fed at step ``t``."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, t, 0xF112]))
    shape = (spec.B, spec.S, spec.Hkv, spec.d)
    return _bf16_normals(rng, shape), _bf16_normals(rng, shape)


def tiny_fill() -> FillSpec:
    return FillSpec(B=2, K=4, F=(4, 2, 1, 1, 1), V=4096, dtype="f32", T=1.0, C=0.5, Hq=4, Hkv=2,
                    d=64, L=37, recipe="gauss", name="tiny-cache-fill-B2-K4-S9-V4096-f32")


def llama3_fill() -> FillSpec:
    """The draft-attention tree (K = 4, F = (8,4,2,1,1), chains of 4 nodes) over
    the Llama-3 vocabulary: 16 sequences, 16 branches each."""
    return FillSpec(B=16, K=4, F=(8, 4, 2, 1, 1), V=128256, dtype="bf16", T=1.0, C=0.5, Hq=32,
                    Hkv=8, d=64, L=2048, name="llama3-cache-fill-B16-K4-S16-V128256-bf16-C0.5")


# ---------------------------------------------------------------------------
# Token trees for multi-candidate verification
# ---------------------------------------------------------------------------
@dataclass
class TreeSpec:
    """A batch of token trees: level-order nodes where each node of depth d has
    branching[d] children; per node a target and a draft logit row."""
    B: int
    V: int
    dtype: str
    T: float
    branching: tuple
    recipe: str = "zipf"       # "zipf" (-1.1 ln rank + N(0, .3^2)) or "gauss" (N(0, 2^2))
    draft_noise: float = 1.0   # draft = target + N(0, draft_noise^2)
    name: str = ""

    @property
    def N(self) -> int:
        return len(tree_shape(self.branching))


def tree_shape(branching) -> np.ndarray:
    """Parent indices of a level-order tree: the root (-1) has branching[0]
    children, each node of depth d has branching[d] children."""
    parent, level = [], [-1]
    for nb in branching:
        nxt = []
        for u in level:
            for _ in range(nb):
                parent.append(u)
                nxt.append(len(parent) - 1)
        level = nxt
    return np.asarray(parent, dtype=np.int32)


def tree_logits(spec: TreeSpec, seed: int, seqs=None):
    """Target and draft logits [len(seqs), N+1, V] (float32, or bf16 bits):
    row 0 at the root, row m+1 after node m; generated per (seed, sequence)."""
    seqs = range(spec.B) if seqs is None else seqs
    N1 = spec.N + 1
    tgt, dft = [], []
    for b in seqs:
        rng = np.random.default_rng(np.random.SeedSequence([seed, b, 0x7733]))
        if spec.recipe == "zipf":
            zt, zd = _zipf_rows(rng, N1, spec.V, 1.1, 0.3, spec.draft_noise)
        else:
            zt, zd = _gauss_rows(rng, N1, spec.V, 2.0, spec.draft_noise)
        if spec.dtype != "f32":
            zt, zd = f32_to_bf16_bits(zt), f32_to_bf16_bits(zd)
        tgt.append(zt)
        dft.append(zd)
    return np.stack(tgt), np.stack(dft)


def tree_uniforms(seed: int, rnd: int, B: int, N: int):
    """``u_acc[B, N]`` and ``u_bonus[B]`` of a tree walk (Philox counters
    (round, sequence, SLOT_TREE, node) and (round, sequence, SLOT_TREE_BONUS, 0))."""
    key = (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    b = np.arange(B, dtype=np.uint32)[:, None]

    def draw(kind, n):
        j = np.arange(n, dtype=np.uint32)[None, :]
        ctr = np.stack(np.broadcast_arrays(np.uint32(rnd & 0xFFFFFFFF), b, np.uint32(kind), j), axis=-1)
        return uniforms_from_bits(philox4x32_10(ctr, key)[..., 0])
    return draw(SLOT_TREE, N), draw(SLOT_TREE_BONUS, 1)[:, 0].copy()


def tiny_tree() -> TreeSpec:
    return TreeSpec(B=3, V=4096, dtype="f32", T=1.0, branching=(3, 2, 1), recipe="gauss",
                    draft_noise=0.8, name="tiny-tree-B3-N15-V4096-f32")


def llama3_tree(B: int = 32) -> TreeSpec:
    """A 28-node tree (4 candidates at the root, 2 below each, then chains)
    over the Llama-3 vocabulary."""
    return TreeSpec(B=B, V=128256, dtype="bf16", T=1.0, branching=(4, 2, 1, 1),
                    name=f"llama3-tree-B{B}-N28-V128256-bf16")


# ---------------------------------------------------------------------------
# Token histories for the miss fallback
# ---------------------------------------------------------------------------
def backup_uniforms(seed: int, rnd: int, B: int, K: int) -> np.ndarray:
    """``u_rand[B, K]``: the uniforms of the random-token backup (Philox counter
    (round, sequence, SLOT_BACKUP, position))."""
    key = (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    b = np.arange(B, dtype=np.uint32)[:, None]
    j = np.arange(K, dtype=np.uint32)[None, :]
    ctr = np.stack(np.broadcast_arrays(np.uint32(rnd & 0xFFFFFFFF), b, np.uint32(SLOT_BACKUP), j),
                   axis=-1)
    return uniforms_from_bits(philox4x32_10(ctr, key)[..., 0])


@dataclass
class HistorySpec:
    """Shape and value recipe of the histories a miss-fallback call reads."""
    B: int
    K: int
    V: int
    L_min: int                 # history lengths ~ uniform integers in [L_min, L_max]
    L_max: int
    cap: int = 0               # row capacity (>= L_max; 0: L_max)
    n: int = 3                 # n-gram length
    zipf_slope: float = 1.1    # fresh tokens: P(rank r) ~ r^-slope over a seeded permutation
    copy_prob: float = 0.3     # a span repeats an earlier span with this chance
    span_min: int = 4          # span lengths ~ uniform integers in [span_min, span_max]
    span_max: int = 32
    miss_rate: float = 0.3     # each sequence missed the cache with this chance
    name: str = ""


@dataclass
class HistoryInputs:
    spec: HistorySpec
    hist: np.ndarray           # [B, cap] int32, zero past hist_len
    hist_len: np.ndarray       # [B] int32
    slot: np.ndarray           # [B] int32: -1 for a miss, else a cache slot
    u_rand: np.ndarray         # [B, K] float32


def _zipf_sampler(rng, V: int, slope: float):
    perm = rng.permutation(V).astype(np.int32)
    w = np.arange(1, V + 1, dtype=np.float64) ** -slope
    cdf = np.cumsum(w)
    cdf /= cdf[-1]

    def draw(n):
        r = np.minimum(np.searchsorted(cdf, rng.random(n), side="right"), V - 1)
        return perm[r]
    return draw


def make_histories(spec: HistorySpec, seed: int = 0, rnd: int = 0) -> HistoryInputs:
    """Seeded histories: fresh Zipf tokens in spans, each span after the first
    copying an earlier span of the same sequence with chance ``copy_prob``."""
    rng = np.random.default_rng(seed)
    cap = spec.cap or spec.L_max
    draw = _zipf_sampler(rng, spec.V, spec.zipf_slope)
    lens = rng.integers(spec.L_min, spec.L_max + 1, size=spec.B).astype(np.int32)
    hist = np.zeros((spec.B, cap), np.int32)
    for b in range(spec.B):
        L = int(lens[b])
        h = draw(L).astype(np.int32)
        pos = 0
        while pos < L:
            s = int(rng.integers(spec.span_min, spec.span_max + 1))
            s = min(s, L - pos)
            if pos >= s and rng.random() < spec.copy_prob:
                src = int(rng.integers(0, pos - s + 1))
                h[pos:pos + s] = h[src:src + s]
            pos += s
        hist[b, :L] = h
    slot = np.where(rng.random(spec.B) < spec.miss_rate, -1,
                    rng.integers(0, 64, size=spec.B)).astype(np.int32)
    return HistoryInputs(spec, hist, lens, slot, backup_uniforms(seed, rnd, spec.B, spec.K))


def qwen3_histories(B: int = 256) -> HistorySpec:
    """The large-batch Qwen-3 round's batch and vocabulary, with prompt+generation
    histories of 1-8 Ki tokens and the 3-gram backup."""
    return HistorySpec(B=B, K=4, V=151936, L_min=1024, L_max=8192, n=3,
                       name=f"qwen3-ngram-backup-B{B}-K4-V151936-L1k-8k-n3")


def tiny_histories() -> HistorySpec:
    return HistorySpec(B=48, K=6, V=50, L_min=0, L_max=700, cap=704, n=2, zipf_slope=0.8,
                       copy_prob=0.4, span_min=2, span_max=9, miss_rate=0.7,
                       name="tiny-ngram-backup-B48-K6-V50-L0-700-n2")


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("math", "np", "dataclass", "field")]

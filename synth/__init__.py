"""Seeded synthetic inputs for the verification step.

This module is shared by the tests, the benchmark and the oracle scripts. It
only draws random numbers and packs them into the layouts the library reads;
it holds none of the verification arithmetic (no temperature softmax, no
accept test, no residual, no argmax). Draft tokens are drawn here because the
draft model is outside the verification step: the generator plays the draft
model's sampler (a Gumbel-max draw), or plants the draft token by construction.

Workload shapes follow the pages' descriptions:
  * "aiengineeringfromscratch.com - Speculative decoding and EAGLE-3",
    section on the Leviathan rejection sampler: target distributions
    q_1..q_{N+1}, draft distributions p_1..p_N, one uniform per accept test;
  * "devpost.com - phoenix", section "What it does": greedy verification, whose
    output must equal the target's own argmax decode.

Layouts (all C-contiguous):
  target logits  [B, K+1, V]   bf16 bits (uint16) or float32
  draft  logits  [B, K,   V]   same dtype as target
  draft tokens   [B, K]        int32 in [0, V)
  uniforms       [B, K+1]      float32 in [0, 1)
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BF16 = "bf16"
F32 = "f32"


# --------------------------------------------------------------------------
# bf16 representation helpers (bit-level packing, not arithmetic of the method)
# --------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round-to-nearest-even), return uint16 bits.

    Non-finite inputs keep their class (inf stays inf, NaN stays a quiet NaN).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    nan = np.isnan(x)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    r[nan] = 0x7FC0
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 values."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def logits_values(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Decode a stored logits array (bf16 bits or float32) to float32 values."""
    if dtype == BF16:
        return bf16_bits_to_f32(arr)
    return np.asarray(arr, dtype=np.float32)


# --------------------------------------------------------------------------
# random streams
# --------------------------------------------------------------------------
def philox_uniforms(shape, seed: int) -> np.ndarray:
    """float32 uniforms in [0, 1) from NumPy's counter-based Philox generator."""
    g = np.random.Generator(np.random.Philox(seed))
    return g.random(shape, dtype=np.float32)


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def gumbel_max_draw(rng: np.random.Generator, scores: np.ndarray) -> np.ndarray:
    """Draft-model sampler: index of max(scores + Gumbel noise) on the last axis.

    `scores` are the draft logits already divided by the draft temperature.
    This is how the synthetic draft model proposes its token; it is not part of
    the verification step and the verifier never calls it.
    """
    g = rng.gumbel(size=scores.shape)
    return np.argmax(scores + g, axis=-1).astype(np.int32)


# --------------------------------------------------------------------------
# cases
# --------------------------------------------------------------------------
@dataclass
class VerifyCase:
    """One batch of verifier inputs plus the recipe that produced it."""

    target: np.ndarray          # [B, K+1, V] uint16 (bf16 bits) or float32
    draft: np.ndarray | None    # [B, K, V] same dtype, None for greedy-only cases
    tokens: np.ndarray          # [B, K] int32
    uniforms: np.ndarray        # [B, K+1] float32
    temperature: float
    dtype: str
    recipe: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return self.target.shape[0]

    @property
    def K(self) -> int:
        return self.target.shape[1] - 1

    @property
    def V(self) -> int:
        return self.target.shape[2]

    def target_values(self) -> np.ndarray:
        return logits_values(self.target, self.dtype)

    def draft_values(self) -> np.ndarray:
        return logits_values(self.draft, self.dtype)


def _store(x32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == BF16:
        return f32_to_bf16_bits(x32)
    return np.ascontiguousarray(x32, dtype=np.float32)


def sampling_case(B: int, K: int, V: int, *, temperature: float, target_std: float,
                  draft_noise_std: float, dtype: str = BF16, seed: int = 0,
                  uniform_seed: int | None = None) -> VerifyCase:
    """Sampling-mode workload.

    target logits ~ N(0, target_std^2) iid; draft logits = target + N(0, draft_noise_std^2)
    (added in float32, then stored in `dtype`); draft token i ~ softmax(draft_i / T)
    drawn with the Gumbel-max trick; uniforms from Philox(uniform_seed).
    """
    rng = _rng(seed)
    zt = rng.normal(0.0, target_std, size=(B, K + 1, V)).astype(np.float32)
    tgt = _store(zt, dtype)
    zt_v = logits_values(tgt, dtype)
    noise = rng.normal(0.0, draft_noise_std, size=(B, K, V)).astype(np.float32)
    drf = _store(zt_v[:, :K, :] + noise, dtype)
    del noise
    zd_v = logits_values(drf, dtype).astype(np.float64)
    tok = np.empty((B, K), np.int32)
    T = float(np.float32(temperature))
    for b in range(B):  # row by row to bound the Gumbel buffer
        tok[b] = gumbel_max_draw(rng, zd_v[b] / T)
    u = philox_uniforms((B, K + 1), seed if uniform_seed is None else uniform_seed)
    return VerifyCase(tgt, drf, tok, u, temperature, dtype,
                      dict(kind="sampling", B=B, K=K, V=V, T=temperature, target_std=target_std,
                           draft_noise_std=draft_noise_std, dtype=dtype, seed=seed,
                           uniform_seed=uniform_seed))


def normal_target(B: int, K: int, V: int, *, target_std: float = 3.0, dtype: str = BF16,
                  seed: int = 0) -> np.ndarray:
    """Target logits [B, K+1, V] ~ N(0, target_std^2) iid, stored in `dtype`,
    unaltered (no clipping, nothing planted): in bf16 the largest values of a
    long row often round to the same value, so argmax ties occur naturally."""
    rng = _rng(seed)
    return _store(rng.normal(0.0, target_std, size=(B, K + 1, V)).astype(np.float32), dtype)


PLANT_VALUE = 16.0      # exactly representable in bf16
CLIP = 14.5             # every other logit is clipped below PLANT_VALUE


def greedy_case(B: int, K: int, V: int, *, alpha: float, target_std: float = 3.0,
                dtype: str = BF16, seed: int = 0) -> VerifyCase:
    """Greedy workload with planted acceptance.

    Target logits ~ N(0, target_std^2), clipped to [-CLIP, CLIP]; at every
    position one token g (uniform) is raised to PLANT_VALUE, so the argmax is g
    by construction without the generator computing one. Draft token i equals
    g_i with probability alpha, else a uniformly random other token.
    """
    rng = _rng(seed)
    z = np.clip(rng.normal(0.0, target_std, size=(B, K + 1, V)), -CLIP, CLIP).astype(np.float32)
    g = rng.integers(0, V, size=(B, K + 1))
    bi, pi = np.meshgrid(np.arange(B), np.arange(K + 1), indexing="ij")
    z[bi, pi, g] = PLANT_VALUE
    tgt = _store(z, dtype)
    hit = rng.random((B, K)) < alpha
    other = (g[:, :K] + 1 + rng.integers(0, V - 1, size=(B, K))) % V
    tok = np.where(hit, g[:, :K], other).astype(np.int32)
    u = philox_uniforms((B, K + 1), seed)
    return VerifyCase(tgt, None, tok, u, 0.0, dtype,
                      dict(kind="greedy", B=B, K=K, V=V, alpha=alpha, target_std=target_std,
                           dtype=dtype, seed=seed, planted=g.astype(np.int32)))


# --------------------------------------------------------------------------
# draft trees
# --------------------------------------------------------------------------
@dataclass
class TreeCase:
    """One batch of greedy tree-verification inputs.

    target [B, N+1, V] (row 0: after the committed prefix, row 1 + i: after
    node i), parents [B, N] int32 (topological order, -1 = root child),
    tokens [B, N] int32.
    """

    target: np.ndarray
    parents: np.ndarray
    tokens: np.ndarray
    dtype: str
    recipe: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return self.target.shape[0]

    @property
    def N(self) -> int:
        return self.parents.shape[1]

    @property
    def V(self) -> int:
        return self.target.shape[2]

    def target_values(self) -> np.ndarray:
        return logits_values(self.target, self.dtype)


def tree_parents(branching) -> np.ndarray:
    """Parents of a full tree in breadth-first order: `branching[d]` children
    per node at depth d (the lesson's exercise uses [2, 2, 2]: 14 nodes)."""
    par, level = [], [-1]
    for k in branching:
        nxt = []
        for p in level:
            for _ in range(int(k)):
                nxt.append(len(par))
                par.append(p)
        level = nxt
    return np.asarray(par, np.int32)


def random_parents(rng: np.random.Generator, N: int) -> np.ndarray:
    """A random tree in topological order: parent of node i uniform in [-1, i)."""
    return np.asarray([rng.integers(-1, i) for i in range(N)], np.int32)


def tree_case(B: int, V: int, *, branching=(2, 2, 2), N: int | None = None, alpha: float = 0.7,
              target_std: float = 3.0, distinct: bool = True, dtype: str = BF16,
              seed: int = 0) -> TreeCase:
    """Greedy tree workload with planted argmaxes.

    Shape: the full tree `branching` (same for every row), or, with N given,
    a random topological tree per row. Every target row gets one planted
    maximum g (as in greedy_case). Each sibling group (the children of one
    row) carries g of that row with probability alpha at a random child;
    the other children take tokens other than g. distinct=True keeps sibling
    tokens distinct (a top-k proposal); False draws them independently, so
    duplicate siblings occur.
    """
    rng = _rng(seed)
    if N is None:
        par = np.tile(tree_parents(branching), (B, 1))
    else:
        par = np.stack([random_parents(rng, N) for _ in range(B)]) if N else np.zeros((B, 0), np.int32)
    N = par.shape[1]
    z = np.clip(rng.normal(0.0, target_std, size=(B, N + 1, V)), -CLIP, CLIP).astype(np.float32)
    g = rng.integers(0, V, size=(B, N + 1))
    bi, pi = np.meshgrid(np.arange(B), np.arange(N + 1), indexing="ij")
    z[bi, pi, g] = PLANT_VALUE
    tok = np.empty((B, N), np.int32)
    for b in range(B):
        for r in range(N + 1):                       # sibling group under row r
            kids = [i for i in range(N) if par[b, i] == r - 1]
            if not kids:
                continue
            if distinct:
                pool = (g[b, r] + 1 + rng.permutation(V - 1)[:len(kids)]) % V
            else:
                pool = (g[b, r] + 1 + rng.integers(0, V - 1, size=len(kids))) % V
            for j, i in enumerate(kids):
                tok[b, i] = pool[j]
            if distinct:
                if rng.random() < alpha:
                    tok[b, kids[rng.integers(0, len(kids))]] = g[b, r]
            else:
                hit = rng.random(len(kids)) < alpha
                for j, i in enumerate(kids):
                    if hit[j]:
                        tok[b, i] = g[b, r]
    return TreeCase(_store(z, dtype), par.astype(np.int32), tok, dtype,
                    dict(kind="tree_greedy", B=B, V=V, N=N, branching=list(branching) if N is None
                         else None, alpha=alpha, distinct=distinct, target_std=target_std,
                         dtype=dtype, seed=seed, planted=g.astype(np.int32)))


# --------------------------------------------------------------------------
# paged KV cache state
# --------------------------------------------------------------------------
@dataclass
class KVCase:
    """Paged KV-cache bookkeeping state before one commit/rollback.

    block_table [B, max_blocks] int32 (-1 unused), seq_lens [B] int32,
    prov_blocks [B, P] int32 (provisional blocks holding slots 0..K),
    free_stack [num_blocks] int32 with free_top live entries at the bottom,
    num_accepted [B] int32 in [0, K]. Block contents are not held here.
    """

    block_table: np.ndarray
    seq_lens: np.ndarray
    prov_blocks: np.ndarray
    free_stack: np.ndarray
    free_top: int
    num_accepted: np.ndarray
    num_blocks: int
    block_size: int
    K: int
    recipe: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return self.seq_lens.shape[0]

    @property
    def P(self) -> int:
        return self.prov_blocks.shape[1]

    @property
    def max_blocks(self) -> int:
        return self.block_table.shape[1]


def kv_case(B: int, K: int, *, block_size: int = 16, prefix_lo: int = 512, prefix_hi: int = 4096,
            spare_blocks: int = 64, num_accepted: np.ndarray | None = None, seed: int = 0,
            seq_lens: np.ndarray | None = None, max_blocks: int | None = None) -> KVCase:
    """Random paged-cache state: prefix lengths ~ U[prefix_lo, prefix_hi], blocks
    assigned from a shuffled pool, ceil((K+1)/block_size) provisional blocks per
    row, and `spare_blocks` extra free blocks."""
    rng = _rng(seed)
    if seq_lens is None:
        seq_lens = rng.integers(prefix_lo, prefix_hi + 1, size=B).astype(np.int32)
    seq_lens = np.asarray(seq_lens, np.int32)
    P = -(-(K + 1) // block_size)
    used = [-(-int(s) // block_size) for s in seq_lens]
    need_max = max(-(-(int(s) + K + 1) // block_size) for s in seq_lens) if B else 1
    if max_blocks is None:
        max_blocks = need_max
    num_blocks = sum(used) + B * P + B * (-(-(K + 1) // block_size) + 1) + spare_blocks
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = np.full((B, max_blocks), -1, np.int32)
    pos = 0
    for b in range(B):
        bt[b, :used[b]] = perm[pos:pos + used[b]]
        pos += used[b]
    prov = perm[pos:pos + B * P].reshape(B, P).copy()
    pos += B * P
    free = np.full(num_blocks, -1, np.int32)
    nfree = num_blocks - pos
    free[:nfree] = perm[pos:]
    if num_accepted is None:
        num_accepted = rng.integers(0, K + 1, size=B).astype(np.int32)
    return KVCase(bt, seq_lens.copy(), prov, free, nfree, np.asarray(num_accepted, np.int32),
                  num_blocks, block_size, K,
                  dict(kind="kv", B=B, K=K, block_size=block_size, prefix_lo=prefix_lo,
                       prefix_hi=prefix_hi, spare_blocks=spare_blocks, seed=seed))


# --------------------------------------------------------------------------
# the named workloads (shapes and distributions from the pages' workloads)
# --------------------------------------------------------------------------
def pr1_case(step: int, steps: int = 1000) -> VerifyCase:
    """B=1, K=4, V=32000 float32; target ~ N(0, 2^2), draft = target + N(0, 0.5^2),
    T = 1.0; uniforms U(0,1) from Philox seed 0 (row `step` of a [steps, K+1] draw).
    Step `step` of the 1000 independent steps."""
    c = sampling_case(1, 4, 32000, temperature=1.0, target_std=2.0, draft_noise_std=0.5,
                      dtype=F32, seed=1_000_003 + step)
    c.uniforms = philox_uniforms((steps, 5), 0)[step:step + 1].copy()
    c.recipe["uniform_seed"] = 0
    c.recipe["step"] = step
    return c

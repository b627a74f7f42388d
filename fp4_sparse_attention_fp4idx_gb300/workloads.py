"""Seeded synthetic inputs for the fused FP4 indexer pre-pass.

This module only draws inputs: it holds none of the method's arithmetic, and
both the CUDA path and the CPU oracle consume what it returns.  Everything is
generated on the host with numpy's PCG64 (identical streams on x86-64 and
aarch64); bf16 tensors are returned as uint16 bit patterns, rounded from fp32
draws with torch's CPU fp32->bf16 conversion.

Workload shapes follow the pages' indexer shapes (head_dim 128, rope_dim 64,
group 32, kv_block 64; H = 32 or 64 query heads; DeepSeek / GLM-style decode,
MTP and prefill batches).  The RoPE tables are the caller-side cos/sin cache,
fp32 [max_pos, 32], theta = pos * base^(-2i/64) evaluated in double.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

HEAD_DIM = 128
ROPE_HALF = 32
KV_BLOCK = 64
PAGE_BYTES = KV_BLOCK * 68
ROPE_NEOX = 0
ROPE_INTERLEAVED = 1

# E2M1 midpoints and the group anchor 6 used to build exact-tie rows.
_MID_PATTERN = [6.0, 0.25, -0.25, 0.75, -0.75, 1.25, -1.25, 1.75, -1.75,
                2.5, -2.5, 3.5, -3.5, 5.0, -5.0]


def to_bf16_bits(x) -> np.ndarray:
    """fp32/fp64 array -> bf16 bit patterns (uint16), via torch CPU."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def rope_tables(max_pos: int, base: float = 10000.0):
    """cos/sin fp32 [max_pos, 32]: theta(p, i) = p * base^(-2i/64)."""
    i = np.arange(ROPE_HALF, dtype=np.float64)
    inv_freq = base ** (-2.0 * i / (2 * ROPE_HALF))
    theta = np.arange(max_pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.cos(theta).astype(np.float32), np.sin(theta).astype(np.float32)


def _normal_bf16(rng, shape, chunk_rows: int = 1 << 22) -> np.ndarray:
    """N(0,1) bf16 bits, drawn in chunks of rows to bound host memory."""
    shape = tuple(shape)
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    step = chunk_rows * HEAD_DIM
    for s in range(0, n, step):
        e = min(n, s + step)
        out[s:e] = to_bf16_bits(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


def midpoint_group_values(scale_pow2: int) -> np.ndarray:
    """32 values 2^k * {6, +-0.25, +-0.75, ..., +-5, 0...}: with anchor 6*2^k
    the group's scale is exactly 2^k, so every listed value sits on an exact
    E2M1 midpoint after scaling."""
    v = np.zeros(32, np.float64)
    v[:len(_MID_PATTERN)] = _MID_PATTERN
    return v * (2.0 ** scale_pow2)


def midpoint_key_row() -> np.ndarray:
    """A 128-element key row whose exact midpoints survive RMSNorm when gamma
    is 1: row = 8 * p where each group of p holds the 15 midpoint/anchor
    values plus integer fillers (11, 11, 10, 10 sixes; a one in groups 2, 3).
    The squares of p add up to 2048 exactly, so the mean square of the row is
    64 * 2048 / 128 = 1024 = 4^5 and the normalised row is exactly p / 4."""
    p = np.zeros((4, 32), np.float64)
    sixes = [11, 11, 10, 10]
    ones = [0, 0, 1, 1]
    for g in range(4):
        p[g, :15] = _MID_PATTERN
        p[g, 15:15 + sixes[g]] = 6.0
        p[g, 15 + sixes[g]:15 + sixes[g] + ones[g]] = 1.0
    assert float((p * p).sum()) == 2048.0
    return (8.0 * p).reshape(-1)


def subnormal_bf16(rng, n: int) -> np.ndarray:
    """Random bf16 subnormals: exponent field 0, mantissa 1..127, random sign."""
    mant = rng.integers(1, 128, size=n, dtype=np.uint16)
    sign = rng.integers(0, 2, size=n, dtype=np.uint16) << 15
    return (mant | sign).astype(np.uint16)


@dataclass
class Workload:
    name: str
    T: int
    H: int
    rope_style: int
    q: np.ndarray            # uint16 [T,H,128]
    w: np.ndarray            # uint16 [T,H]
    k: np.ndarray            # uint16 [T,128]
    gamma: np.ndarray        # uint16 [128]
    eps: float
    positions: np.ndarray    # int64 [T]
    cos: np.ndarray          # f32 [max_pos,32]
    sin: np.ndarray          # f32 [max_pos,32]
    slot_mapping: np.ndarray  # int64 [T]
    num_blocks: int
    cache_init: np.ndarray   # uint8 [num_blocks, 4352] sentinel bytes
    notes: dict = field(default_factory=dict)

    @property
    def max_pos(self) -> int:
        return int(self.cos.shape[0])


def _sentinel_cache(rng, num_blocks: int) -> np.ndarray:
    return rng.integers(0, 256, size=(num_blocks, PAGE_BYTES), dtype=np.uint8)


def _gamma(rng) -> np.ndarray:
    return to_bf16_bits(1.0 + 0.1 * rng.standard_normal(HEAD_DIM))


def make_tiny(gamma_one: bool = False) -> Workload:
    """T=8, H=32, NeoX, seed 0.  Token 1 all zeros, token 2 bf16 subnormals,
    token 3 exact E2M1 midpoints at position 0 (RoPE is the identity there).
    With gamma_one the key midpoints survive RMSNorm too."""
    rng = np.random.Generator(np.random.PCG64(0))
    T, H = 8, 32
    q = _normal_bf16(rng, (T, H, HEAD_DIM))
    k = _normal_bf16(rng, (T, HEAD_DIM))
    q[1] = 0
    k[1] = 0
    q[2] = subnormal_bf16(rng, H * HEAD_DIM).reshape(H, HEAD_DIM)
    k[2] = subnormal_bf16(rng, HEAD_DIM)
    for h in range(H):
        q[3, h] = to_bf16_bits(np.concatenate(
            [midpoint_group_values(h - 16 + g) for g in range(4)]))
    k[3] = to_bf16_bits(midpoint_key_row())
    gamma = to_bf16_bits(np.ones(HEAD_DIM)) if gamma_one else _gamma(rng)
    if gamma_one:
        _gamma(rng)  # keep the stream aligned with the gamma~N case
    positions = rng.integers(0, 4096, size=T, dtype=np.int64)
    positions[3] = 0
    cos, sin = rope_tables(4096)
    w = _normal_bf16(rng, (T, H))
    num_blocks = 4
    slots = rng.permutation(num_blocks * KV_BLOCK)[:T].astype(np.int64)
    cache = _sentinel_cache(rng, num_blocks)
    return Workload("tiny_gamma1" if gamma_one else "tiny", T, H, ROPE_NEOX,
                    q, w, k, gamma, 1e-6, positions, cos, sin, slots,
                    num_blocks, cache)


def make_decode() -> Workload:
    """T=256, H=64, interleaved RoPE, seed 1.  Rows ~N(0,1) times a per-row
    factor from {1, 40, 1e-3}; positions U[0,131072); 4096 blocks; distinct
    random slots with 10% set to -1."""
    rng = np.random.Generator(np.random.PCG64(1))
    T, H = 256, 64
    fac = np.array([1.0, 40.0, 1e-3])
    qf = rng.standard_normal((T, H, HEAD_DIM)) * fac[rng.integers(0, 3, (T, H, 1))]
    kf = rng.standard_normal((T, HEAD_DIM)) * fac[rng.integers(0, 3, (T, 1))]
    q = to_bf16_bits(qf)
    k = to_bf16_bits(kf)
    gamma = _gamma(rng)
    max_pos = 131072
    positions = rng.integers(0, max_pos, size=T, dtype=np.int64)
    cos, sin = rope_tables(max_pos)
    w = _normal_bf16(rng, (T, H))
    num_blocks = 4096
    slots = rng.choice(num_blocks * KV_BLOCK, size=T, replace=False).astype(np.int64)
    slots[rng.random(T) < 0.10] = -1
    cache = _sentinel_cache(rng, num_blocks)
    return Workload("decode", T, H, ROPE_INTERLEAVED, q, w, k, gamma, 1e-6,
                    positions, cos, sin, slots, num_blocks, cache)


def make_prefill() -> Workload:
    """T=8192, H=64, NeoX, positions 0..8191, seed 2.  N(0,1) with 1% of the
    entries (Bernoulli mask) scaled by 50 before the bf16 cast; 8192 blocks,
    the tokens filling 128 consecutive blocks from a seeded start block."""
    rng = np.random.Generator(np.random.PCG64(2))
    T, H = 8192, 64

    def draw(shape):
        x = rng.standard_normal(shape, dtype=np.float32)
        x[rng.random(shape, dtype=np.float32) < 0.01] *= 50.0
        return to_bf16_bits(x)

    q = draw((T, H, HEAD_DIM))
    k = draw((T, HEAD_DIM))
    gamma = _gamma(rng)
    positions = np.arange(T, dtype=np.int64)
    cos, sin = rope_tables(T)
    w = _normal_bf16(rng, (T, H))
    num_blocks = 8192
    start = int(rng.integers(0, num_blocks - T // KV_BLOCK + 1))
    slots = start * KV_BLOCK + np.arange(T, dtype=np.int64)
    cache = _sentinel_cache(rng, num_blocks)
    return Workload("prefill", T, H, ROPE_NEOX, q, w, k, gamma, 1e-6,
                    positions, cos, sin, slots, num_blocks, cache)


def make_large_prefill(T: int = 65536) -> Workload:
    """T=65536, H=64, NeoX, positions 0..T-1, N(0,1), seed 3; 16384 blocks,
    token t -> block perm[t // 64], offset t % 64 (perm a random permutation
    of the blocks).  A smaller T keeps the same recipe for quick runs."""
    rng = np.random.Generator(np.random.PCG64(3))
    H = 64
    q = _normal_bf16(rng, (T, H, HEAD_DIM))
    k = _normal_bf16(rng, (T, HEAD_DIM))
    gamma = _gamma(rng)
    positions = np.arange(T, dtype=np.int64)
    cos, sin = rope_tables(T)
    w = _normal_bf16(rng, (T, H))
    num_blocks = 16384
    perm = rng.permutation(num_blocks).astype(np.int64)
    t = np.arange(T, dtype=np.int64)
    slots = perm[t // KV_BLOCK] * KV_BLOCK + t % KV_BLOCK
    cache = _sentinel_cache(rng, num_blocks)
    return Workload("large_prefill" if T == 65536 else f"large_prefill_T{T}",
                    T, H, ROPE_NEOX, q, w, k, gamma, 1e-6, positions, cos,
                    sin, slots, num_blocks, cache)


def make_mtp() -> Workload:
    """1024 sequences x next_n=4 (T=4096), H=32, interleaved RoPE, seed 4.
    Per-sequence base position U[0,65536) plus offsets 0..3; Laplace(0,1)
    bf16; 65536 blocks; each sequence's one or two pages drawn without reuse
    from a random block permutation; 5% of slots set to -1."""
    rng = np.random.Generator(np.random.PCG64(4))
    S, NN, H = 1024, 4, 32
    T = S * NN
    q = to_bf16_bits(rng.laplace(0.0, 1.0, (T, H, HEAD_DIM)))
    k = to_bf16_bits(rng.laplace(0.0, 1.0, (T, HEAD_DIM)))
    gamma = _gamma(rng)
    base = rng.integers(0, 65536, size=S, dtype=np.int64)
    positions = (base[:, None] + np.arange(NN, dtype=np.int64)[None, :]).reshape(-1)
    max_pos = 65536 + NN - 1
    cos, sin = rope_tables(max_pos)
    w = _normal_bf16(rng, (T, H))
    num_blocks = 65536
    perm = iter(rng.permutation(num_blocks).astype(np.int64).tolist())
    slots = np.empty(T, np.int64)
    for s in range(S):
        table = {}
        for j in range(NN):
            p = int(positions[s * NN + j])
            lb = p // KV_BLOCK
            if lb not in table:
                table[lb] = next(perm)
            slots[s * NN + j] = table[lb] * KV_BLOCK + p % KV_BLOCK
    slots[rng.random(T) < 0.05] = -1
    cache = _sentinel_cache(rng, num_blocks)
    return Workload("mtp", T, H, ROPE_INTERLEAVED, q, w, k, gamma, 1e-6,
                    positions, cos, sin, slots, num_blocks, cache)


def make_random(T: int, H: int, rope_style: int, seed: int, max_pos: int = 512,
                num_blocks: int | None = None, skip_frac: float = 0.1,
                scales=(1.0, 40.0, 1e-3)) -> Workload:
    """Small generic case: per-row scales, random positions, random distinct
    slots with a fraction skipped."""
    rng = np.random.Generator(np.random.PCG64(seed))
    fac = np.asarray(scales, np.float64)
    qf = rng.standard_normal((T, H, HEAD_DIM)) * fac[rng.integers(0, len(fac), (T, H, 1))]
    kf = rng.standard_normal((T, HEAD_DIM)) * fac[rng.integers(0, len(fac), (T, 1))]
    q = to_bf16_bits(qf)
    k = to_bf16_bits(kf)
    gamma = _gamma(rng)
    positions = rng.integers(0, max_pos, size=T, dtype=np.int64)
    cos, sin = rope_tables(max_pos)
    w = _normal_bf16(rng, (T, H))
    if num_blocks is None:
        num_blocks = max(1, (2 * T + KV_BLOCK - 1) // KV_BLOCK)
    slots = rng.choice(num_blocks * KV_BLOCK, size=T, replace=False).astype(np.int64)
    slots[rng.random(T) < skip_frac] = -1
    cache = _sentinel_cache(rng, num_blocks)
    return Workload(f"random_T{T}_H{H}_s{rope_style}_{seed}", T, H, rope_style,
                    q, w, k, gamma, 1e-6, positions, cos, sin, slots,
                    num_blocks, cache)


CONFIGS = {
    "tiny": make_tiny,
    "decode": make_decode,
    "prefill": make_prefill,
    "large_prefill": make_large_prefill,
    "mtp": make_mtp,
}


def make(name: str) -> Workload:
    if name == "tiny_gamma1":
        return make_tiny(gamma_one=True)
    return CONFIGS[name]()


# ------------------------------------------------------------------ scorer
@dataclass
class ScorerWorkload:
    """Inputs of the FP4 paged MQA-logits scorer: packed queries with their
    exponent words and fp32 head weights (what the query half of the pre-pass
    emits) and a paged index-K cache (what the key half writes), drawn
    directly as bytes."""
    name: str
    batch: int
    next_n: int
    H: int
    max_context: int
    q_fp4: np.ndarray         # uint8 [batch*next_n, H, 64]
    q_scale: np.ndarray       # uint8 [batch*next_n, H, 4]
    weights: np.ndarray       # f32 [batch*next_n, H]
    kv_cache: np.ndarray      # uint8 [num_blocks, 4352]
    block_table: np.ndarray   # int32 [batch, pages]; -1 past each context
    context_lens: np.ndarray  # int32 [batch]
    notes: dict = field(default_factory=dict)

    @property
    def num_blocks(self) -> int:
        return int(self.kv_cache.shape[0])

    def rows_of(self, seqs) -> "ScorerWorkload":
        """The same inputs restricted to the given sequences (for sampled
        oracle checks at full size); the cache is shared, not copied."""
        seqs = np.asarray(seqs)
        rows = (seqs[:, None] * self.next_n + np.arange(self.next_n)[None, :]).reshape(-1)
        return ScorerWorkload(self.name, len(seqs), self.next_n, self.H, self.max_context,
                              self.q_fp4[rows], self.q_scale[rows], self.weights[rows],
                              self.kv_cache, self.block_table[seqs], self.context_lens[seqs],
                              dict(self.notes, rows=rows))


def make_scorer(name: str, batch: int, next_n: int, H: int, context_lens, max_context: int,
                seed: int, exp_range=(118, 135), spare_blocks: int = 3,
                extremes: bool = False) -> ScorerWorkload:
    """Uniform random payload nibbles (every E2M1 code, both signs, -0
    included), exponent bytes uniform in exp_range, weights ~ N(0,1) *
    (H*128)^-1/2.  Pages are a random permutation of the pool; block-table
    entries past a sequence's context are -1 and must never be read.  With
    `extremes`, some key groups are all-zero at the floor exponent 1 (what the
    pre-pass writes for a zero group), some sit at exponent 1 with non-zero
    codes (values 2^-127 .. 6*2^-126), and some use exponents 150..160."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = np.asarray(context_lens, dtype=np.int32)
    assert ctx.shape == (batch,)
    pages_needed = [max(0, -(-int(min(c, max_context)) // KV_BLOCK)) for c in ctx]
    num_blocks = sum(pages_needed) + spare_blocks
    width = max(1, -(-max_context // KV_BLOCK))
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = np.full((batch, width), -1, dtype=np.int32)
    at = 0
    for b, n in enumerate(pages_needed):
        bt[b, :n] = perm[at:at + n]
        at += n
    lo, hi = exp_range
    cache = rng.integers(0, 256, size=(num_blocks, PAGE_BYTES), dtype=np.uint8)
    cache[:, KV_BLOCK * 64:] = rng.integers(lo, hi + 1, size=(num_blocks, KV_BLOCK * 4),
                                            dtype=np.uint8)
    rows = batch * next_n
    q_fp4 = rng.integers(0, 256, size=(rows, H, 64), dtype=np.uint8)
    q_scale = rng.integers(lo, hi + 1, size=(rows, H, 4), dtype=np.uint8)
    weights = (rng.standard_normal((rows, H)) / np.sqrt(H * HEAD_DIM)).astype(np.float32)
    if extremes:
        n_tok = num_blocks * KV_BLOCK
        for kind in range(3):
            picks = rng.choice(n_tok, size=max(1, n_tok // 16), replace=False)
            for tok in picks:
                page, o = divmod(int(tok), KV_BLOCK)
                g = int(rng.integers(0, 4))
                payload = cache[page, o * 64 + 16 * g:o * 64 + 16 * g + 16]
                if kind == 0:
                    payload[:] = 0
                    cache[page, KV_BLOCK * 64 + 4 * o + g] = 1
                elif kind == 1:
                    cache[page, KV_BLOCK * 64 + 4 * o + g] = 1
                else:
                    cache[page, KV_BLOCK * 64 + 4 * o + g] = rng.integers(150, 161)
    return ScorerWorkload(name, batch, next_n, H, max_context, q_fp4, q_scale, weights, cache,
                          bt, ctx, {"seed": seed, "exp_range": exp_range,
                                    "extremes": extremes})


def _ragged_lens(rng, batch: int, lo: int, hi: int) -> np.ndarray:
    return rng.integers(lo, hi + 1, size=batch).astype(np.int32)


def make_scorer_decode(batch: int = 128, next_n: int = 4, H: int = 32,
                       max_context: int = 65536, seed: int = 21,
                       name: str = "scorer_decode") -> ScorerWorkload:
    """GLM-5.2-style decode with multi-token prediction: H = 32 index heads,
    next_n = 4 query tokens per sequence, 128 sequences with context lengths
    uniform in [max_context/4, max_context] (about 5.2M cached tokens, 350 MB
    of index-K cache, 134 MB of logits)."""
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    lens = _ragged_lens(rng, batch, max_context // 4, max_context)
    return make_scorer(name, batch, next_n, H, lens, max_context, seed)


SCORER_CONFIGS = {
    # name: (batch, next_n, H, context_lens, max_context, seed, extremes)
    "scorer_tiny": (3, 1, 32, [0, 1, 200], 260, 31, True),
    "scorer_glm_next1": (5, 1, 32, [64, 127, 129, 700, 1000], 1024, 32, True),
    "scorer_glm_next4": (4, 4, 32, [1, 255, 256, 777], 800, 33, False),
    "scorer_dsv_next1": (3, 1, 64, [300, 64, 513], 520, 34, True),
    "scorer_dsv_next2": (3, 2, 64, [128, 5, 640], 700, 35, False),
    "scorer_r96": (2, 3, 32, [450, 200], 450, 36, False),
    "scorer_h128": (2, 1, 128, [333, 129], 384, 37, True),
    # more than 128 query rows per sequence: groups of 128 / H tokens
    "scorer_dsv_next4": (3, 4, 64, [300, 64, 513], 520, 38, True),
    "scorer_h64_next3": (2, 3, 64, [200, 450], 450, 39, False),
    "scorer_h128_next2": (2, 2, 128, [129, 333], 384, 40, True),
    "scorer_h96_next3": (2, 3, 96, [100, 200], 256, 42, False),
    "scorer_h32_next8": (2, 8, 32, [130, 64], 200, 43, False),
}


# Many short sequences: every CTA spans several sequences, so the query
# operand buffers are reused within a launch.
SCORER_MANY = {
    # name: (batch, next_n, H, max_context, seed)
    "scorer_many_short": (900, 4, 32, 130, 81),
    "scorer_many_short_r256": (700, 4, 64, 200, 82),
    "scorer_many_short_r192": (800, 3, 64, 256, 83),
    "scorer_many_short_r96": (900, 3, 32, 200, 84),
}


def make_scorer_config(name: str) -> ScorerWorkload:
    if name == "scorer_decode":
        return make_scorer_decode()
    if name in SCORER_MANY:
        b, n, h, mc, seed = SCORER_MANY[name]
        rng = np.random.Generator(np.random.PCG64(seed + 1000))
        return make_scorer(name, b, n, h, _ragged_lens(rng, b, 0, mc), mc, seed)
    b, n, h, lens, mc, seed, ext = SCORER_CONFIGS[name]
    return make_scorer(name, b, n, h, lens, mc, seed, extremes=ext)


def fp8_sentinel_cache(w: Workload) -> np.ndarray:
    """Seeded sentinel bytes for the FP8 output mode's cache: the same number
    of pages as the workload's FP4 cache, 8448 bytes each."""
    seed = 7919 + 31 * w.T + w.H + sum(map(ord, w.name))
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(0, 256, size=(w.num_blocks, KV_BLOCK * (HEAD_DIM + 4)), dtype=np.uint8)


@dataclass
class PrefillScorerWorkload:
    """Inputs of the FP4 prefill MQA-logits scorer: T query tokens (packed
    queries, exponent words, fp32 head weights) against num_keys consecutive
    keys (key s at page s/64, offset s%64 of the cache), token t over the
    keys [ks[t], ke[t])."""
    name: str
    T: int
    H: int
    num_keys: int
    q_fp4: np.ndarray     # uint8 [T, H, 64]
    q_scale: np.ndarray   # uint8 [T, H, 4]
    weights: np.ndarray   # f32 [T, H]
    kv_cache: np.ndarray  # uint8 [num_blocks, 4352]
    ks: np.ndarray        # int32 [T]
    ke: np.ndarray        # int32 [T]

    @property
    def num_blocks(self) -> int:
        return int(self.kv_cache.shape[0])


def make_prefill_scorer(name: str, T: int, H: int, num_keys: int, seed: int,
                        ranges: str = "causal", exp_range=(118, 135),
                        spare_blocks: int = 2) -> PrefillScorerWorkload:
    """Bytes drawn as in make_scorer.  Key ranges:
      causal  -- a prefill chunk whose T tokens are the last T of the
                 num_keys keys: token t scores keys [0, num_keys - T + t + 1);
      windows -- random ranges [a, b) inside [0, num_keys), some empty;
      edges   -- ranges that need clamping or are empty: negative starts,
                 ends past num_keys, a == b, a > b, tile-boundary ends."""
    rng = np.random.Generator(np.random.PCG64(seed))
    nb = -(-num_keys // KV_BLOCK) + spare_blocks
    lo, hi = exp_range
    cache = rng.integers(0, 256, size=(nb, PAGE_BYTES), dtype=np.uint8)
    cache[:, KV_BLOCK * 64:] = rng.integers(lo, hi + 1, size=(nb, KV_BLOCK * 4), dtype=np.uint8)
    q_fp4 = rng.integers(0, 256, size=(T, H, 64), dtype=np.uint8)
    q_scale = rng.integers(lo, hi + 1, size=(T, H, 4), dtype=np.uint8)
    weights = (rng.standard_normal((T, H)) / np.sqrt(H * HEAD_DIM)).astype(np.float32)
    t = np.arange(T)
    if ranges == "causal":
        ks = np.zeros(T, np.int64)
        ke = num_keys - T + t + 1
    elif ranges == "windows":
        a = rng.integers(0, num_keys, T)
        b = rng.integers(0, num_keys + 1, T)
        ks, ke = np.minimum(a, b), np.maximum(a, b)
        ke[::7] = ks[::7]  # some empty ranges
    elif ranges == "edges":
        cands = [(-5, 10), (0, num_keys + 100), (-3, num_keys + 3), (7, 7), (50, 20),
                 (128, 256), (127, 129), (num_keys - 1, num_keys), (num_keys, num_keys + 5),
                 (-10, -2), (64, 65), (0, 1)]
        pick = [cands[i % len(cands)] for i in range(T)]
        ks = np.array([c[0] for c in pick], np.int64)
        ke = np.array([c[1] for c in pick], np.int64)
    else:
        raise ValueError(ranges)
    return PrefillScorerWorkload(name, T, H, num_keys, q_fp4, q_scale, weights, cache,
                                 ks.astype(np.int32), ke.astype(np.int32))


PREFILL_SCORER_CONFIGS = {
    # name: (T, H, num_keys, seed, ranges)
    "prefill_tiny_causal": (5, 32, 70, 61, "causal"),
    "prefill_h32_causal": (300, 32, 300, 62, "causal"),
    "prefill_h64_windows": (77, 64, 1000, 63, "windows"),
    "prefill_h64_edges": (24, 64, 300, 64, "edges"),
    "prefill_h128_causal": (33, 128, 500, 65, "causal"),
    "prefill_h128_windows": (9, 128, 260, 66, "windows"),
    "prefill_h96_edges": (13, 96, 129, 67, "edges"),
}


def make_prefill_scorer_config(name: str) -> PrefillScorerWorkload:
    T, H, nk, seed, ranges = PREFILL_SCORER_CONFIGS[name]
    return make_prefill_scorer(name, T, H, nk, seed, ranges)


def make_prefill_scorer_chunk(T: int = 4096, H: int = 64, num_keys: int = 16384,
                              seed: int = 71) -> PrefillScorerWorkload:
    """A DeepSeek-shaped prefill chunk: H = 64 index heads, the last 4096
    tokens of a 16384-token prompt, causal key ranges (about 12K keys per
    token, 268 MB of logits)."""
    return make_prefill_scorer("prefill_chunk", T, H, num_keys, seed, "causal")



@dataclass
class IndexerE2E:
    """Raw bf16 inputs of the whole indexer path for `batch` sequences of
    `ctx` tokens: every token's key (to be normalised, rotated, quantised and
    stored through slot_mapping into shuffled pages), and the last next_n
    tokens' queries and head weights.  Keys of sequence b are tokens
    b*ctx .. b*ctx + ctx - 1 at positions 0 .. ctx-1; its query token j sits
    at position ctx - next_n + j."""
    name: str
    batch: int
    ctx: int
    next_n: int
    H: int
    rope_style: int
    k: np.ndarray            # bf16 bits [batch*ctx, 128]
    k_positions: np.ndarray  # int64 [batch*ctx]
    slot_mapping: np.ndarray  # int64 [batch*ctx]
    gamma: np.ndarray        # bf16 bits [128]
    eps: float
    q: np.ndarray            # bf16 bits [batch*next_n, H, 128]
    w: np.ndarray            # bf16 bits [batch*next_n, H]
    q_positions: np.ndarray  # int64 [batch*next_n]
    cos: np.ndarray
    sin: np.ndarray
    num_blocks: int
    block_table: np.ndarray  # int32 [batch, ctx/64]
    context_lens: np.ndarray  # int32 [batch]


def make_indexer_e2e(batch: int = 4, ctx: int = 2048, next_n: int = 4, H: int = 32,
                     rope_style: int = ROPE_NEOX, seed: int = 91) -> IndexerE2E:
    """GLM-5.2-shaped indexer inputs (H = 32, D = 128, kv_block 64): N(0,1)
    bf16 keys, queries and head weights, gamma ~ 1 + 0.1 N(0,1), each
    sequence's pages a random permutation of the pool."""
    rng = np.random.Generator(np.random.PCG64(seed))
    assert ctx % KV_BLOCK == 0
    pages = ctx // KV_BLOCK
    nb = batch * pages
    perm = rng.permutation(nb).astype(np.int64)
    bt = perm.reshape(batch, pages).astype(np.int32)
    tok = np.arange(batch * ctx)
    b, s = tok // ctx, tok % ctx
    slots = perm.reshape(batch, pages)[b, s // KV_BLOCK] * KV_BLOCK + s % KV_BLOCK
    cos, sin = rope_tables(ctx)
    qpos = np.tile(np.arange(ctx - next_n, ctx, dtype=np.int64), batch)
    return IndexerE2E(f"indexer_e2e_b{batch}_c{ctx}_n{next_n}_h{H}", batch, ctx, next_n, H,
                      rope_style, _normal_bf16(rng, (batch * ctx, HEAD_DIM)),
                      s.astype(np.int64), slots.astype(np.int64), _gamma(rng), 1e-6,
                      _normal_bf16(rng, (batch * next_n, H, HEAD_DIM)),
                      _normal_bf16(rng, (batch * next_n, H)), qpos, cos, sin, nb, bt,
                      np.full(batch, ctx, np.int32))

"""Pins of the oracle's FP4 paged MQA-logits scorer: closed-form cases built
byte by byte, the ReLU and head weighting, the page indirection, the context
padding and exact rational arithmetic.  Sources: "[HIP] Add FP4 output mode to
indexer_qk_rope_quant_and_cache" (aiter PR 5484), Verification (the FP4
scorer reads the pre-pass's bytes); "[ROCm][Perf] Enabled FP4Indexer for
DSV4" (vLLM PR 42908), Code Review (scaled E2M1 dot products of packed
queries and keys with their block scales)."""
from fractions import Fraction as Fr

import numpy as np

import oracle

GRID = [Fr(0), Fr(1, 2), Fr(1), Fr(3, 2), Fr(2), Fr(3), Fr(4), Fr(6)]


def pack(nibbles, exps):
    """128 nibbles + 4 exponent bytes -> (64 payload bytes, 4 bytes); the
    even element goes to the low nibble."""
    n = np.asarray(nibbles, np.uint8)
    return (n[0::2] | (n[1::2] << 4)).astype(np.uint8), np.asarray(exps, np.uint8)


def put_slot(cache, slot, payload, exps):
    b, o = divmod(slot, 64)
    cache[b, o * 64:o * 64 + 64] = payload
    cache[b, 4096 + 4 * o:4096 + 4 * o + 4] = exps


def value(nib, e):
    v = GRID[nib & 7] * Fr(2) ** (e - 127)
    return -v if nib & 8 else v


def one_hot(d, nib, e=127):
    n = np.zeros(128, np.uint8)
    n[d] = nib
    return pack(n, [e] * 4)


def test_single_element_closed_form():
    """q has 1.0 at dim 5, k has 3.0 (1.5 * 2^1) at dim 5: score 3, weight
    0.5, logit 1.5; a negated key gives a negative score, so ReLU -> 0."""
    qp, qe = one_hot(5, 2)
    kp, ke = one_hot(5, 3, 128)
    kpn, _ = one_hot(5, 3 | 8, 128)
    cache = np.zeros((2, 4352), np.uint8)
    put_slot(cache, 0, kp, ke)
    put_slot(cache, 1, kpn, ke)
    out, st = oracle.paged_mqa_logits(qp[None, None], qe[None, None],
                                      np.array([[0.5]], np.float32), cache,
                                      np.array([[0]], np.int32), np.array([2], np.int32), 1, 4)
    assert st == 0
    assert out[0, 0] == 1.5 and out[0, 1] == 0.0
    assert np.isneginf(out[0, 2]) and np.isneginf(out[0, 3])


def test_heads_weighted_relu_sum():
    """Two heads: scores +2 and -4; only the positive one counts, weighted."""
    qp0, qe = one_hot(0, 4)        # 2.0
    qp1, _ = one_hot(0, 6 | 8)     # -4.0
    kp, ke = one_hot(0, 2)         # 1.0
    cache = np.zeros((1, 4352), np.uint8)
    put_slot(cache, 0, kp, ke)
    q = np.stack([qp0, qp1])[None]
    qs = np.stack([qe, qe])[None]
    out, _ = oracle.paged_mqa_logits(q, qs, np.array([[0.25, 10.0]], np.float32), cache,
                                     np.array([[0]], np.int32), np.array([1], np.int32), 1, 1)
    assert out[0, 0] == 0.5


def test_group_exponents_scale_the_score():
    """A 1.0 * 1.0 product in group g scales by 2^(eq-127) * 2^(ek-127)."""
    for g, eq, ek in ((0, 130, 120), (2, 100, 140), (3, 127, 127)):
        nq = np.zeros(128, np.uint8)
        nq[32 * g + 7] = 2
        nk = np.zeros(128, np.uint8)
        nk[32 * g + 7] = 2
        eqs = [127] * 4
        eks = [127] * 4
        eqs[g], eks[g] = eq, ek
        qp, qe = pack(nq, eqs)
        kp, ke = pack(nk, eks)
        cache = np.zeros((1, 4352), np.uint8)
        put_slot(cache, 0, kp, ke)
        out, _ = oracle.paged_mqa_logits(qp[None, None], qe[None, None],
                                         np.ones((1, 1), np.float32), cache,
                                         np.array([[0]], np.int32), np.array([1], np.int32), 1, 1)
        assert out[0, 0] == np.float32(2.0 ** (eq + ek - 254))


def test_page_indirection_and_sequences():
    """Token s of sequence b lives at page block_table[b, s/64], offset s%64;
    every row of a sequence (next_n rows) sees that sequence's tokens."""
    rng = np.random.Generator(np.random.PCG64(3))
    B, next_n, ctx = 2, 2, 130
    cache = np.zeros((8, 4352), np.uint8)
    bt = np.array([[5, 2, 7], [0, 6, 1]], np.int32)
    expect = np.full((B * next_n, 192), -np.inf, np.float32)
    q = np.zeros((B * next_n, 1, 64), np.uint8)
    qs = np.full((B * next_n, 1, 4), 127, np.uint8)
    for r in range(B * next_n):
        q[r, 0] = one_hot(r, 2)[0]  # 1.0 at dim r
    for b in range(B):
        for s in range(ctx):
            code = int(rng.integers(1, 8))
            n = np.zeros(128, np.uint8)
            n[b * next_n:(b + 1) * next_n] = code  # the dims the rows of b read
            kp, ke = pack(n, [127] * 4)
            put_slot(cache, int(bt[b, s // 64]) * 64 + s % 64, kp, ke)
            for j in range(next_n):
                expect[b * next_n + j, s] = float(GRID[code])
    out, st = oracle.paged_mqa_logits(q, qs, np.ones((B * next_n, 1), np.float32), cache, bt,
                                      np.array([ctx, ctx], np.int32), next_n, 192)
    assert st == 0 and np.array_equal(out, expect)


def test_bad_page_reported():
    cache = np.zeros((1, 4352), np.uint8)
    q = np.zeros((1, 1, 64), np.uint8)
    qs = np.full((1, 1, 4), 127, np.uint8)
    out, st = oracle.paged_mqa_logits(q, qs, np.ones((1, 1), np.float32), cache,
                                      np.array([[3]], np.int32), np.array([2], np.int32), 1, 2)
    assert st == -1 and np.all(np.isneginf(out))


def test_random_case_exact_rational():
    """Random codes and exponents: the oracle equals the exact rational value
    rounded to fp32 (within 1 ulp for the double accumulation)."""
    rng = np.random.Generator(np.random.PCG64(4))
    B, next_n, H, ctx = 2, 2, 3, 70
    nbl = 4
    cache = rng.integers(0, 256, (nbl, 4352), dtype=np.uint8)
    cache[:, 4096:] = rng.integers(118, 137, (nbl, 256), dtype=np.uint8)
    bt = np.array([[1, 3], [2, 0]], np.int32)
    q = rng.integers(0, 256, (B * next_n, H, 64), dtype=np.uint8)
    qs = rng.integers(118, 137, (B * next_n, H, 4), dtype=np.uint8)
    w = rng.standard_normal((B * next_n, H)).astype(np.float32)
    out, st = oracle.paged_mqa_logits(q, qs, w, cache, bt, np.array([ctx, ctx - 9], np.int32),
                                      next_n, 72)
    assert st == 0
    for (t, s) in [(0, 0), (1, 5), (1, 64), (0, 69), (2, 0), (3, 60), (2, 33)]:
        b = t // next_n
        page = int(bt[b, s // 64])
        o = s % 64
        kv = []
        for d in range(128):
            byte = int(cache[page, o * 64 + d // 2])
            nib = byte >> 4 if d % 2 else byte & 15
            kv.append(value(nib, int(cache[page, 4096 + 4 * o + d // 32])))
        acc = Fr(0)
        for h in range(H):
            dot = Fr(0)
            for d in range(128):
                byte = int(q[t, h, d // 2])
                nib = byte >> 4 if d % 2 else byte & 15
                dot += value(nib, int(qs[t, h, d // 32])) * kv[d]
            if dot > 0:
                acc += Fr(float(w[t, h])) * dot
        want = np.float32(float(acc))
        got = out[t, s]
        assert abs(int(np.float32(got).view(np.int32)) - int(want.view(np.int32))) <= 1, (t, s)
    assert np.all(np.isneginf(out[2:, ctx - 9:]))


# ----------------------------------------------------------------- prefill
def exact_logit(q, qs, w, cache, t, page, o):
    """sum_h w * max(0, q . k) by exact rationals, rounded once to fp32."""
    kv = []
    for d in range(128):
        byte = int(cache[page, o * 64 + d // 2])
        nib = byte >> 4 if d % 2 else byte & 15
        kv.append(value(nib, int(cache[page, 4096 + 4 * o + d // 32])))
    acc = Fr(0)
    for h in range(q.shape[1]):
        dot = Fr(0)
        for d in range(128):
            byte = int(q[t, h, d // 2])
            nib = byte >> 4 if d % 2 else byte & 15
            dot += value(nib, int(qs[t, h, d // 32])) * kv[d]
        if dot > 0:
            acc += Fr(float(w[t, h])) * dot
    return np.float32(float(acc))


def test_prefill_ranges_and_exact_values():
    """The prefill scorer: token t scores the consecutive keys s in
    [ks[t], ke[t]) (key s in page s/64 at offset s%64), -inf elsewhere;
    sampled logits equal the exact rational value (within 1 ulp)."""
    rng = np.random.Generator(np.random.PCG64(44))
    T, H, nk = 6, 3, 150
    cache = rng.integers(0, 256, (3, 4352), dtype=np.uint8)
    cache[:, 4096:] = rng.integers(118, 137, (3, 256), dtype=np.uint8)
    q = rng.integers(0, 256, (T, H, 64), dtype=np.uint8)
    qs = rng.integers(118, 137, (T, H, 4), dtype=np.uint8)
    w = rng.standard_normal((T, H)).astype(np.float32)
    ks = np.array([0, 10, 64, 149, 30, 5], np.int32)
    ke = np.array([150, 11, 128, 150, 30, 2], np.int32)   # t=4, t=5: empty ranges
    out, st = oracle.mqa_logits_prefill(q, qs, w, cache, ks, ke, nk)
    assert st == 0 and out.shape == (T, nk)
    for t in range(T):
        inside = (np.arange(nk) >= ks[t]) & (np.arange(nk) < ke[t])
        assert np.all(np.isneginf(out[t, ~inside])) and np.all(np.isfinite(out[t, inside]))
    for (t, s) in [(0, 0), (0, 149), (1, 10), (2, 64), (2, 127), (3, 149), (0, 65)]:
        want = exact_logit(q, qs, w, cache, t, s // 64, s % 64)
        got = np.float32(out[t, s])
        assert abs(int(got.view(np.int32)) - int(want.view(np.int32))) <= 1, (t, s)


def test_prefill_single_element_closed_form():
    """q = 1.0 at dim 9 for one head of weight 2; key 70 (page 1, offset 6)
    holds 1.5 * 2^2 = 6 at dim 9, key 71 holds -6: logits 12 and 0."""
    qp, qe = one_hot(9, 2)
    kp, ke_ = one_hot(9, 3, 129)
    kn, _ = one_hot(9, 3 | 8, 129)
    cache = np.zeros((2, 4352), np.uint8)
    put_slot(cache, 70, kp, ke_)
    put_slot(cache, 71, kn, ke_)
    out, _ = oracle.mqa_logits_prefill(qp[None, None], qe[None, None],
                                       np.array([[2.0]], np.float32), cache,
                                       np.array([70], np.int32), np.array([72], np.int32), 80)
    assert out[0, 70] == 12.0 and out[0, 71] == 0.0
    assert np.all(np.isneginf(out[0, :70])) and np.all(np.isneginf(out[0, 72:]))


def test_prefill_matches_paged_scorer_on_identity_table():
    """With every token's range the whole chunk, the prefill scorer is the
    paged scorer of one sequence whose block table is the identity (key s in
    page s/64) and whose next_n is the token count."""
    rng = np.random.Generator(np.random.PCG64(45))
    T, H, nk = 5, 32, 200
    pages = -(-nk // 64)
    cache = rng.integers(0, 256, (pages, 4352), dtype=np.uint8)
    cache[:, 4096:] = rng.integers(118, 137, (pages, 256), dtype=np.uint8)
    q = rng.integers(0, 256, (T, H, 64), dtype=np.uint8)
    qs = rng.integers(118, 137, (T, H, 4), dtype=np.uint8)
    w = rng.standard_normal((T, H)).astype(np.float32)
    pre, st = oracle.mqa_logits_prefill(q, qs, w, cache, np.zeros(T, np.int32),
                                        np.full(T, nk, np.int32), nk)
    assert st == 0
    paged, st = oracle.paged_mqa_logits(q, qs, w, cache, np.arange(pages, dtype=np.int32)[None],
                                        np.array([nk], np.int32), T, nk)
    assert st == 0
    assert np.array_equal(pre.view(np.uint32), paged.view(np.uint32))

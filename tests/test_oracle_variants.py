"""Pins of the oracle's stated variants of the pre-pass: the optional
Walsh-Hadamard rotation before quantisation ("DeepSeek-V4 FP4: fused_compress
FP4 scatter + rmsnorm_rope_rotate FP4 KV-cache kernel" (aiter PR 4029),
Changes: RMSNorm + RoPE + optional Hadamard rotate + FP4 quant) and the key
RoPE at the first position of a compressed group ("dsv4.1: RoPE and FP4
packing kernels" (sglang PR 39656), Summary and Verification: compress ratios
1, 2, 4).  Each pin checks the oracle against something other than itself:
exact closed forms, a library matrix, or a sign pattern fixed by the
transform's definition."""
import numpy as np
import pytest

import oracle
from fp4_sparse_attention_fp4idx_gb300 import workloads as wl

NORM = np.float32(1.0 / np.sqrt(128.0))


def sylvester(n: int) -> np.ndarray:
    """The Sylvester Hadamard matrix, entry (i, j) = (-1)^popcount(i & j),
    built by the doubling recursion (not by the transform under test)."""
    h = np.ones((1, 1), np.int64)
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def bf16_of(x) -> np.ndarray:
    return wl.to_bf16_bits(np.asarray(x, np.float32))


def f32_of(bits) -> np.ndarray:
    return wl.bf16_bits_to_f32(bits)


def test_sylvester_entries_closed_form():
    h = sylvester(128)
    i, j = np.meshgrid(np.arange(128), np.arange(128), indexing="ij")
    pc = np.vectorize(lambda v: bin(v).count("1"))(i & j)
    assert np.array_equal(h, np.where(pc % 2 == 0, 1, -1))


def test_hadamard_one_hot_rows():
    """e_i maps to row i of H times rn32(1/sqrt(128)), rounded to bf16: one
    fp32 product per element, no sums, so the value is exact."""
    h = sylvester(128)
    for i in (0, 1, 5, 64, 127):
        x = np.zeros(128, np.float32)
        x[i] = 1.0
        got = f32_of(oracle.hadamard_row(bf16_of(x)))
        want = f32_of(bf16_of(h[i].astype(np.float32) * NORM))
        assert np.array_equal(got, want), i


def test_hadamard_small_integers_exact():
    """Integer inputs keep every butterfly sum exact in fp32, so the result
    is bf16(rn32(H x) * rn32(1/sqrt(128))) with H x from the matrix."""
    rng = np.random.Generator(np.random.PCG64(5))
    h = sylvester(128)
    for _ in range(20):
        x = rng.integers(-40, 41, 128).astype(np.float32)
        got = f32_of(oracle.hadamard_row(bf16_of(x)))
        hx = (h @ x.astype(np.int64)).astype(np.float32)
        want = f32_of(bf16_of(hx * NORM))
        assert np.array_equal(got, want)


def test_hadamard_matches_fp64_matrix_product():
    """General bf16 rows: within one bf16 ulp of the fp64 product with
    scipy's Hadamard matrix, and equal to its bf16 rounding almost always
    (the fp32 butterflies differ from exact arithmetic only by rounding)."""
    scipy_linalg = pytest.importorskip("scipy.linalg")
    hm = scipy_linalg.hadamard(128).astype(np.float64)
    rng = np.random.Generator(np.random.PCG64(6))
    same = total = 0
    for _ in range(200):
        x = f32_of(bf16_of(rng.standard_normal(128) * 10.0 ** rng.uniform(-3, 3)))
        exact = hm @ x.astype(np.float64) / np.sqrt(128.0)
        got = f32_of(oracle.hadamard_row(bf16_of(x))).astype(np.float64)
        ulp = np.abs(f32_of(bf16_of(exact)).astype(np.float64)) * 2.0 ** -7
        assert np.all(np.abs(got - exact) <= ulp + 1e-38)
        same += int(np.sum(got == f32_of(bf16_of(exact))))
        total += 128
    assert same / total > 0.97


def test_hadamard_twice_is_identity():
    """H/sqrt(128) is orthogonal and symmetric: applied twice it returns the
    row up to the roundings.  The intermediate's bf16 rounding (at most 2^-9
    relative per element) passes through the orthogonal second transform as
    an error vector of norm <= 2^-9 |x|_2; the final rounding adds 2^-9 |y|."""
    rng = np.random.Generator(np.random.PCG64(7))
    for _ in range(50):
        x = f32_of(bf16_of(rng.standard_normal(128)))
        y = f32_of(oracle.hadamard_row(oracle.hadamard_row(bf16_of(x))))
        bound = 2.0 ** -9 * np.linalg.norm(x.astype(np.float64)) * 1.01 + 2.0 ** -8 * np.abs(x)
        assert np.all(np.abs(y - x) <= bound)


def _sign_bits(payload: np.ndarray) -> np.ndarray:
    """Sign bits of the 128 nibbles of a 64-byte payload (even element in the
    low nibble)."""
    nib = np.empty(128, np.uint8)
    nib[0::2] = payload & 0x0F
    nib[1::2] = payload >> 4
    return (nib >> 3) & 1


def test_query_rotation_sign_pattern():
    """A one-hot query at position 0 (RoPE is the identity there) rotates to
    +-v/sqrt(128) in every dimension, with the signs of row i of H; every
    code is then the same non-zero magnitude."""
    cos, sin = wl.rope_tables(4)
    h = sylvester(128)
    for i in (3, 77):
        q = np.zeros((1, 1, 128), np.float32)
        q[0, 0, i] = 4.0
        qf, qs, _, st = oracle.q_rope_pack_weights(bf16_of(q), bf16_of(np.ones((1, 1))),
                                                   np.zeros(1, np.int64), cos, sin, 0,
                                                   hadamard=True)
        assert st == 0
        signs = _sign_bits(qf[0, 0])
        assert np.array_equal(signs, (h[i] < 0).astype(np.uint8))
        mags = np.concatenate([qf[0, 0] & 7, (qf[0, 0] >> 4) & 7])
        assert np.all(mags == mags[0]) and mags[0] != 0
        qf0, _, _, _ = oracle.q_rope_pack_weights(bf16_of(q), bf16_of(np.ones((1, 1))),
                                                  np.zeros(1, np.int64), cos, sin, 0)
        nz = np.count_nonzero(np.concatenate([qf0[0, 0] & 15, qf0[0, 0] >> 4]))
        assert nz == 1  # without the rotation one element stays non-zero


def test_key_rotation_sign_pattern():
    """A one-hot key (gamma 1) normalises to sqrt(128) e_i, which rotates to
    +-1 in every dimension with the signs of row i of H."""
    cos, sin = wl.rope_tables(4)
    h = sylvester(128)
    gamma = bf16_of(np.ones(128))
    for i in (0, 100):
        k = np.zeros((1, 128), np.float32)
        k[0, i] = 3.0
        cache = np.zeros((1, wl.PAGE_BYTES), np.uint8)
        st = oracle.k_norm_rope_pack_store(bf16_of(k), gamma, 1e-6, np.zeros(1, np.int64), cos,
                                           sin, 0, np.array([5], np.int64), cache, hadamard=True)
        assert st == 0
        payload = cache[0, 5 * 64:6 * 64]
        assert np.array_equal(_sign_bits(payload), (h[i] < 0).astype(np.uint8))
        mags = np.concatenate([payload & 7, (payload >> 4) & 7])
        assert np.all(mags == mags[0]) and mags[0] != 0


@pytest.mark.parametrize("ratio", [2, 4])
def test_compress_ratio_uses_group_first_position(ratio):
    """Key position p takes the RoPE of p - p % ratio: positions inside the
    first group rotate like position 0 (the identity), and every position
    matches the uncompressed call at the group's first position."""
    rng = np.random.Generator(np.random.PCG64(8 + ratio))
    cos, sin = wl.rope_tables(64)
    T = 24
    k = wl._normal_bf16(rng, (T, 128))
    gamma = wl._gamma(rng)
    pos = np.arange(T, dtype=np.int64) + 3
    slots = np.arange(T, dtype=np.int64)
    got = np.zeros((1, wl.PAGE_BYTES), np.uint8)
    oracle.k_norm_rope_pack_store(k, gamma, 1e-6, pos, cos, sin, 0, slots, got,
                                  compress_ratio=ratio)
    first = np.zeros((1, wl.PAGE_BYTES), np.uint8)
    oracle.k_norm_rope_pack_store(k, gamma, 1e-6, pos - pos % ratio, cos, sin, 0, slots, first)
    assert np.array_equal(got, first)
    plain = np.zeros((1, wl.PAGE_BYTES), np.uint8)
    oracle.k_norm_rope_pack_store(k, gamma, 1e-6, pos, cos, sin, 0, slots, plain)
    moved = [t for t in range(T) if pos[t] % ratio]
    differs = [not np.array_equal(got[0, 64 * t:64 * t + 64], plain[0, 64 * t:64 * t + 64])
               for t in moved]
    assert sum(differs) >= len(moved) - 1
    ident = np.zeros((1, wl.PAGE_BYTES), np.uint8)
    small = np.arange(T, dtype=np.int64) % ratio  # all in the first group
    oracle.k_norm_rope_pack_store(k, gamma, 1e-6, small, cos, sin, 0, slots, ident,
                                  compress_ratio=ratio)
    zero = np.zeros((1, wl.PAGE_BYTES), np.uint8)
    oracle.k_norm_rope_pack_store(k, gamma, 1e-6, np.zeros(T, np.int64), cos, sin, 0, slots,
                                  zero)
    assert np.array_equal(ident, zero)

"""Pins of the oracle's FP8 output mode ("[HIP] Add FP4 output mode to
indexer_qk_rope_quant_and_cache" (aiter PR 5484), Summary and API: the FP8
contract the FP4 mode extends, whose per-(token, head) query scale is folded
into the head weights).  E4M3 (e4m3fn) codes with one power-of-two scale per
128-element row.  Each pin checks the oracle against torch's float8_e4m3fn
conversion, exact rational arithmetic or a closed form."""
from fractions import Fraction as Fr

import numpy as np
import pytest
import torch

import oracle
from fp4_sparse_attention_fp4idx_gb300 import workloads as wl


def torch_e4m3_bytes(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def test_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = np.array([oracle.e4m3_to_f32(c) for c in codes], np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], want[~nan])
    assert oracle.e4m3_to_f32(0x7E) == 448.0 and oracle.e4m3_to_f32(1) == 2.0 ** -9


def test_encode_matches_torch_in_range():
    """Random values across the whole range, every code value, every exact
    midpoint between neighbouring codes (ties to the even mantissa), both
    signs and signed zeros: byte-equal to torch's conversion."""
    rng = np.random.Generator(np.random.PCG64(11))
    finite = np.array([oracle.e4m3_to_f32(c) for c in range(127)], np.float64)
    mids = (finite[:-1] + finite[1:]) / 2.0
    vals = np.concatenate([
        finite, mids, rng.uniform(0, 448, 3000), np.exp2(rng.uniform(-14, 8.8, 3000)),
        [0.0, 2.0 ** -11, 2.0 ** -10, 3 * 2.0 ** -11, 440.0, 447.99],
    ]).astype(np.float32)
    vals = vals[vals <= 448.0]
    vals = np.concatenate([vals, -vals, [-0.0]]).astype(np.float32)
    got = np.array([oracle.f32_to_e4m3(v) for v in vals], np.uint8)
    assert np.array_equal(got, torch_e4m3_bytes(vals))


def test_encode_saturates_above_448():
    for v in (448.5, 465.0, 1e6, 3.0e38):
        assert oracle.f32_to_e4m3(v) == 0x7E
        assert oracle.f32_to_e4m3(-v) == 0xFE


def ceil_pow2_exponent(t: Fr) -> int:
    e = 0
    while Fr(2) ** e < t:
        e += 1
    while Fr(2) ** (e - 1) >= t:
        e -= 1
    return e


def test_row_exponent_exact():
    """e is the biased exponent of ceil_pow2(max(rn32(amax/448), 2^-126)),
    checked with exact rationals; every code then lies in [-448, 448] and the
    row's largest magnitude maps into (224, 448], so its code decodes to a
    value in [224, 448] (224 itself after rounding down), unless the floor
    acts."""
    rng = np.random.Generator(np.random.PCG64(12))
    for trial in range(300):
        scale = 10.0 ** rng.uniform(-30, 30)
        row = wl.to_bf16_bits(rng.standard_normal(128) * scale)
        codes, e = oracle.fp8_quant_row(row)
        x = wl.bf16_bits_to_f32(row)
        amax = float(np.max(np.abs(x)))
        t = Fr(float(np.float32(amax) / np.float32(448.0)))
        t = max(t, Fr(2) ** -126)
        assert e - 127 == ceil_pow2_exponent(t), trial
        dec = np.array([oracle.e4m3_to_f32(c) for c in codes], np.float64)
        top = np.max(np.abs(dec))
        assert 224.0 <= top <= 448.0 or e == 1


def test_row_codes_are_nearest():
    """Each code is the E4M3 value nearest to x * 2^(127-e) (exact product),
    within half a spacing; ties were pinned against torch above."""
    rng = np.random.Generator(np.random.PCG64(13))
    for _ in range(50):
        row = wl.to_bf16_bits(rng.standard_normal(128) * 3.0)
        codes, e = oracle.fp8_quant_row(row)
        x = wl.bf16_bits_to_f32(row).astype(np.float64) * 2.0 ** (127 - e)
        assert np.array_equal(codes, torch_e4m3_bytes(x.astype(np.float32)))


def test_all_zero_row_floor():
    codes, e = oracle.fp8_quant_row(np.zeros(128, np.uint16))
    assert e == 1 and np.all(codes == 0)


def test_key_slot_closed_form():
    """gamma 1 and a constant row normalise to ones; at position 0 RoPE is
    the identity; amax 1 gives scale ceil_pow2(1/448) = 2^-8, so every code
    is 256 = 1.0 * 2^8 (0x78) and the fp32 scale 2^-8 sits at 8192 + 4o."""
    cos, sin = wl.rope_tables(4)
    k = wl.to_bf16_bits(np.full((1, 128), 5.0, np.float32))
    gamma = wl.to_bf16_bits(np.ones(128, np.float32))
    cache = np.full((2, oracle.FP8_PAGE_BYTES), 0xAB, np.uint8)
    st = oracle.k_norm_rope_fp8_store(k, gamma, 1e-6, np.zeros(1, np.int64), cos, sin, 0,
                                      np.array([64 + 9], np.int64), cache)
    assert st == 0
    page = cache[1]
    assert np.all(page[9 * 128:10 * 128] == 0x78)
    assert page[8192 + 36:8192 + 40].view(np.float32)[0] == 2.0 ** -8
    untouched = np.ones(oracle.FP8_PAGE_BYTES, bool)
    untouched[9 * 128:10 * 128] = False
    untouched[8192 + 36:8192 + 40] = False
    assert np.all(page[untouched] == 0xAB) and np.all(cache[0] == 0xAB)


def test_query_weight_folds_scale():
    """H = 32: weight = w * 2^-6 * 2^(e-127), one rounding (here exact); the
    codes are the row's codes."""
    cos, sin = wl.rope_tables(4)
    rng = np.random.Generator(np.random.PCG64(14))
    q = wl.to_bf16_bits(rng.standard_normal((2, 32, 128)))
    w = wl.to_bf16_bits(rng.standard_normal((2, 32)))
    qo, wt, st = oracle.q_rope_fp8_weights(q, w, np.zeros(2, np.int64), cos, sin, 0)
    assert st == 0
    for t in range(2):
        for h in (0, 7, 31):
            codes, e = oracle.fp8_quant_row(q[t, h])
            assert np.array_equal(qo[t, h], codes)
            want = np.float32(wl.bf16_bits_to_f32(w[t, h]) * 2.0 ** -6 * 2.0 ** (e - 127))
            assert wt[t, h] == want


def test_dequantised_values_close():
    """Dequantised codes times the row scale stay within E4M3's rounding of
    the input: at most 2^-4 relative (3 mantissa bits), or half the smallest
    subnormal spacing at the row's scale."""
    rng = np.random.Generator(np.random.PCG64(15))
    for _ in range(20):
        row = wl.to_bf16_bits(rng.standard_normal(128))
        codes, e = oracle.fp8_quant_row(row)
        x = wl.bf16_bits_to_f32(row).astype(np.float64)
        dec = np.array([oracle.e4m3_to_f32(c) for c in codes]) * 2.0 ** (e - 127)
        assert np.all(np.abs(dec - x) <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** (e - 127 - 10)))

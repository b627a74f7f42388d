"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: exact
rational arithmetic, a closed form derived by hand, an invariant the pages
state, a hand-derived fixture in tests/golden/, or a library routine.  The
pages: "dsv4.1: RoPE and FP4 packing kernels" (sglang PR 39656) and
"[HIP] Add FP4 output mode to indexer_qk_rope_quant_and_cache" (aiter PR
5484).
"""
from decimal import Decimal, getcontext
from fractions import Fraction as Fr

import numpy as np
import pytest
import torch

import oracle
from fp4_sparse_attention_fp4idx_gb300 import workloads as wl
from tests import golden

GRID = [Fr(0), Fr(1, 2), Fr(1), Fr(3, 2), Fr(2), Fr(3), Fr(4), Fr(6)]


# ----------------------------------------------------------------- helpers
def bf16_value(bits: int) -> float:
    return float(np.array([bits << 16], np.uint32).view(np.float32)[0])


def all_finite_bf16() -> np.ndarray:
    b = np.arange(1 << 16, dtype=np.uint32)
    finite = ((b >> 7) & 0xFF) != 0xFF
    return b[finite].astype(np.uint16)


def threshold_code(v: np.ndarray) -> np.ndarray:
    """E2M1 code of magnitudes v >= 0 from the midpoints of the grid
    {0,.5,1,1.5,2,3,4,6}: a midpoint goes up exactly when the upper code is
    even (0.75, 1.75, 3.5 go up; 0.25, 1.25, 2.5, 5 stay)."""
    return ((v > 0.25).astype(int) + (v >= 0.75) + (v > 1.25) + (v >= 1.75)
            + (v > 2.5) + (v >= 3.5) + (v > 5.0))


def exact_code(v: Fr) -> int:
    """Nearest grid code of an exact rational, ties to the even code."""
    return min(range(8), key=lambda m: (abs(v - GRID[m]), m % 2))


def ceil_log2(x: Fr) -> int:
    j = x.numerator.bit_length() - x.denominator.bit_length()
    while Fr(2) ** j < x:
        j += 1
    while Fr(2) ** (j - 1) >= x:
        j -= 1
    return j


def exact_exponent(amax: Fr) -> int:
    """Biased UE8M0 exponent of ceil_pow2(max(amax/6, 2^-126))."""
    if amax == 0:
        return 1
    return max(127 + ceil_log2(amax / 6), 1)


def ulp_diff_f32(a, b) -> np.ndarray:
    ia = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    ib = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    ia = np.where(ia < 0, -(ia & 0x7FFFFFFF), ia)
    ib = np.where(ib < 0, -(ib & 0x7FFFFFFF), ib)
    return np.abs(ia - ib)


# ------------------------------------------------------- bf16 round trip
def test_bf16_rounding_matches_torch():
    """The bf16 round trips use fp32->bf16 round-to-nearest-even; pinned to
    torch's CPU conversion over random patterns, exact ties and subnormals."""
    rng = np.random.Generator(np.random.PCG64(11))
    bits = rng.integers(0, 1 << 32, size=60000, dtype=np.uint64).astype(np.uint32)
    ties = (rng.integers(0, 1 << 16, size=20000, dtype=np.uint32) << 16) | 0x8000
    sub = rng.integers(0, 1 << 23, size=20000, dtype=np.uint32) | (
        rng.integers(0, 2, size=20000, dtype=np.uint32) << 31)
    allb = np.concatenate([bits, ties, sub])
    allb = allb[((allb >> 23) & 0xFF) < 0xFE]  # finite and no overflow to inf
    x = allb.view(np.float32)
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f32_to_bf16(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, want)


# ------------------------------------------------------------ E2M1 codes
def test_golden_e2m1_values():
    vals = golden.e2m1_rne_values()
    assert len(vals) == 32
    z = np.array([v for v, _ in vals], np.float32)
    n, e = oracle.quant_group(z)
    assert e == 127
    assert [int(x) for x in n] == [x for _, x in vals]


def test_exponent_exhaustive_bf16():
    """For every finite bf16 amax the exponent is the biased exponent of
    ceil_pow2(max(amax/6, 2^-126)) computed exactly; it stays in [1, 253] so
    the [1, 254] clamp never acts (sglang review, index_pack_exponent)."""
    mags = np.unique(all_finite_bf16() & 0x7FFF)
    es = []
    for b in mags:
        a = bf16_value(int(b))
        z = np.zeros(32, np.float32)
        z[7] = -a if (b & 1) else a
        _, e = oracle.quant_group(z)
        assert e == exact_exponent(Fr(a)), (hex(int(b)), a, e)
        es.append(e)
    assert min(es) == 1 and max(es) == 253


def test_codes_exhaustive_bf16():
    """Every finite bf16 value, quantised in a group whose scale is fixed to
    2^j by an anchor 6*2^j, gets the code the grid's midpoints give, for
    every j in the fp32 normal range; signs follow (z<0 and code!=0)."""
    allv = all_finite_bf16()
    vals = (allv.astype(np.uint32) << 16).view(np.float32)
    mag = np.abs(vals.astype(np.float64))
    checked = 0
    for j in range(-126, 126):
        lo, hi = 2.0 ** (j - 4), 6.0 * 2.0 ** j
        sel = vals[(mag <= hi) & ((mag >= lo) | (mag == 0) | (np.arange(vals.size) % 97 == 0)) & (mag <= hi)]
        anchor = np.float32(6.0 * 2.0 ** j)
        pad = (-sel.size) % 31
        zs = np.concatenate([sel, np.zeros(pad, np.float32)]).reshape(-1, 31)
        for row in zs:
            g = np.concatenate([[anchor], row]).astype(np.float32)
            n, e = oracle.quant_group(g)
            assert e == 127 + j
            v = np.abs(row.astype(np.float64)) / 2.0 ** j
            m = threshold_code(v)
            sign = (row < 0) & (m != 0)
            want = m | (sign.astype(int) << 3)
            assert n[0] == 7
            assert np.array_equal(n[1:].astype(int), want), (j, row, n[1:], want)
        checked += sel.size
    assert checked > 300000


def test_group_quant_exact_rational():
    """Whole-group quantisation against exact rational arithmetic on random
    groups across scales (amax, exponent, nearest code with even ties)."""
    rng = np.random.Generator(np.random.PCG64(5))
    for it in range(400):
        s = 2.0 ** rng.integers(-140, 120)
        z = wl.bf16_bits_to_f32(wl.to_bf16_bits(rng.standard_normal(32) * s))
        if it % 7 == 0:
            z[:] = 0
        n, e = oracle.quant_group(z)
        A = max(abs(Fr(float(x))) for x in z)
        assert e == exact_exponent(A)
        scale = Fr(2) ** (e - 127)
        for x, nib in zip(z, n):
            m = exact_code(abs(Fr(float(x))) / scale)
            assert (nib & 7) == m
            assert (nib >> 3) == (1 if (x < 0 and m != 0) else 0)


def test_all_zero_group():
    """An all-zero group: payload 0 and exponent byte 1 (the floor)."""
    r = oracle.quant_pack_row(np.zeros(128, np.uint16))
    assert not r["payload"].any()
    assert list(r["exp"]) == [1, 1, 1, 1]
    # negative zeros too: -0 never survives as a code
    r = oracle.quant_pack_row(np.full(128, 0x8000, np.uint16))
    assert not r["payload"].any() and list(r["exp"]) == [1, 1, 1, 1]


def test_domain_boundary_top_binade():
    """The stage-1 fake-quant dequantises to bf16: for a group amax up to
    6*2^125 (= 1.5*2^127) every dequantised value is finite; above it the
    scale is 2^126 and codes 6, 7 dequantise to 2^128 and 1.5*2^128, which
    overflow.  Inputs that large are outside the finite domain."""
    a = wl.to_bf16_bits(np.array([6.0 * 2.0 ** 125]))[0]
    row = np.zeros(128, np.uint16)
    row[0] = a
    r = oracle.quant_pack_row(row)
    assert list(r["e1"]) == [252, 1, 1, 1] and list(r["e2"]) == [252, 1, 1, 1]
    assert r["payload"][0] == 7
    assert np.isfinite(oracle.dequant(7, 252))
    row[0] = a + 1  # next bf16 above 6*2^125
    r = oracle.quant_pack_row(row)
    assert r["e1"][0] == 253 and np.isinf(oracle.dequant(6, 253))


def test_inverse_scale_equals_division():
    """Multiplying by the exact inverse scale 2^(127-e) equals dividing by
    2^(e-127) in fp32 for every e in [1, 254] (sglang review,
    inv_scale_ue8m0): both are one rounding of the same real number."""
    rng = np.random.Generator(np.random.PCG64(6))
    z = wl.bf16_bits_to_f32(wl.to_bf16_bits(rng.standard_normal(4096) * 2.0 ** rng.integers(-133, 127, 4096)))
    z = z[np.isfinite(z)]
    for e in range(1, 255):
        inv = np.float32(2.0 ** (127 - e))
        sc = np.float32(2.0 ** (e - 127))
        with np.errstate(over="ignore", under="ignore"):
            a = np.abs(z) * inv
            b = np.abs(z) / sc
        assert np.array_equal(a, b), e


# --------------------------------------------------------- two stages/pack
def test_golden_pack_layout():
    row, pay, exps = golden.pack_layout_row()
    r = oracle.quant_pack_row(wl.to_bf16_bits(row))
    assert np.array_equal(r["payload"], pay)
    assert np.array_equal(r["exp"], exps)


def test_two_stage_invariants():
    """Stage 2 re-encodes stage 1 without changing a dequantised value; its
    exponent is e1 or e1-1, the latter exactly when stage 1's largest code
    is 5 (3.0) and the floor does not hold; non-floor groups end with a top
    code of 6 or 7 (sglang review: the two stages need separate scales)."""
    rng = np.random.Generator(np.random.PCG64(7))
    saw_drop = saw_same = 0
    for it in range(3000):
        s = 2.0 ** rng.integers(-135, 100)
        x = rng.standard_normal(128) * s
        if it % 5 == 0:
            x[rng.random(128) < 0.05] *= 50
        row = wl.to_bf16_bits(x)
        r = oracle.quant_pack_row(row)
        nib2 = np.empty(128, np.uint8)
        nib2[0::2] = r["payload"] & 15
        nib2[1::2] = r["payload"] >> 4
        for g in range(4):
            e1, e2 = int(r["e1"][g]), int(r["e2"][g])
            n1 = r["n1"][32 * g:32 * g + 32]
            n2 = nib2[32 * g:32 * g + 32]
            assert e2 == r["exp"][g]
            d1 = [oracle.dequant(int(a), e1) for a in n1]
            d2 = [oracle.dequant(int(a), e2) for a in n2]
            assert np.array_equal(np.array(d1, np.float32), np.array(d2, np.float32))
            top1 = int((n1 & 7).max())
            if e1 > 1 and top1 == 5:
                assert e2 == e1 - 1
                saw_drop += 1
            else:
                assert e2 == e1
                saw_same += 1
            if e1 > 1:
                assert int((n2 & 7).max()) in (6, 7)
            # sign bit only on a non-zero magnitude
            assert not np.any(((n2 & 8) != 0) & ((n2 & 7) == 0))
    assert saw_drop > 50 and saw_same > 50


def test_negative_zero_statistics_sanity():
    """On N(0,1) bf16 values in groups of 32, roughly 5% of the values are
    negative values that quantise to code 0 (sign cleared) and roughly 0.6%
    sit on exact midpoints (aiter, One deliberate deviation: 5.3% and 0.57%
    of 524,288 values, distribution unstated).  A sanity range only."""
    rng = np.random.Generator(np.random.PCG64(8))
    n = 524288
    bits = wl.to_bf16_bits(rng.standard_normal(n))
    vals = wl.bf16_bits_to_f32(bits).reshape(-1, 32)
    negzero = ties = 0
    for g in vals[:8192]:
        nib, e = oracle.quant_group(g)
        v = np.abs(g.astype(np.float64)) / 2.0 ** (e - 127)
        negzero += int(np.sum((g < 0) & ((nib & 7) == 0)))
        ties += int(np.sum(np.isin(v, [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])))
    frac0 = negzero / (8192 * 32)
    fract = ties / (8192 * 32)
    assert 0.02 < frac0 < 0.10, frac0
    assert 0.001 < fract < 0.02, fract


# ---------------------------------------------------------------- RMSNorm
def test_rmsnorm_constant_row_closed_form():
    """x_i = c with c^2 large enough that eps is absorbed: the mean square is
    c^2, r = 1/c exactly, so y == gamma bit for bit."""
    rng = np.random.Generator(np.random.PCG64(9))
    gamma = wl.to_bf16_bits(1 + 0.1 * rng.standard_normal(128))
    for c in (8.0, 16.0, 64.0, 2.0 ** 20, -8.0):
        x = wl.to_bf16_bits(np.full(128, c))
        y = oracle.rmsnorm_row(x, gamma, 1e-6)
        want = gamma if c > 0 else (gamma ^ 0x8000)
        assert np.array_equal(y, want), c


def test_rmsnorm_midpoint_key_row():
    """The midpoint key row (mean square 1024 exactly) normalises to p/4."""
    row = wl.midpoint_key_row()
    y = oracle.rmsnorm_row(wl.to_bf16_bits(row), wl.to_bf16_bits(np.ones(128)), 1e-6)
    assert np.array_equal(wl.bf16_bits_to_f32(y), (row / 32).astype(np.float32))


def test_rmsnorm_eps_inside_sqrt():
    """For a tiny constant row the eps term dominates: y = c*gamma/sqrt(c^2+eps)
    (closed form, double) to within bf16 rounding."""
    rng = np.random.Generator(np.random.PCG64(10))
    gamma = wl.to_bf16_bits(1 + 0.1 * rng.standard_normal(128))
    g = wl.bf16_bits_to_f32(gamma).astype(np.float64)
    for c in (2.0 ** -12, 2.0 ** -9, 1e-3, 3.0):
        cb = float(wl.bf16_bits_to_f32(wl.to_bf16_bits(np.array([c])))[0])
        y = wl.bf16_bits_to_f32(oracle.rmsnorm_row(wl.to_bf16_bits(np.full(128, cb)), gamma, 1e-6))
        want = cb * g / np.sqrt(cb * cb + float(np.float32(1e-6)))
        assert np.all(np.abs(y - want) <= 2.0 ** -7 * np.abs(want)), c


def test_rmsnorm_random_rows_vs_fp64():
    """Random rows across scales (with subnormal and zero rows): within one
    bf16 rounding plus fp32 error of the fp64 formula."""
    rng = np.random.Generator(np.random.PCG64(12))
    gamma = wl.to_bf16_bits(1 + 0.1 * rng.standard_normal(128))
    g = wl.bf16_bits_to_f32(gamma).astype(np.float64)
    for it in range(300):
        # |x| above ~1.8e19 would overflow the fp32 sum of squares (inputs
        # must keep every intermediate finite), so the top scale is 1e15.
        s = [1.0, 40.0, 1e-3, 2.0 ** -130, 1e15][it % 5]
        xb = wl.to_bf16_bits(rng.standard_normal(128) * s)
        x = wl.bf16_bits_to_f32(xb).astype(np.float64)
        y = wl.bf16_bits_to_f32(oracle.rmsnorm_row(xb, gamma, 1e-6)).astype(np.float64)
        want = x * g / np.sqrt(np.mean(x * x) + float(np.float32(1e-6)))
        tol = 2.0 ** -8 * np.abs(want) + 2.0 ** -20 * np.abs(want) + 1e-38
        assert np.all(np.abs(y - want) <= tol), it


# ------------------------------------------------------------------- RoPE
def _distinct_row(rng):
    return wl.to_bf16_bits(rng.standard_normal(128))


@pytest.mark.parametrize("style", [wl.ROPE_NEOX, wl.ROPE_INTERLEAVED])
def test_rope_identity_and_quarter_turn(style):
    """cos=1, sin=0 is the identity; cos=0, sin=1 maps (a, b) -> (-b, a)
    with NeoX pairs (i, i+32) or interleaved pairs (2i, 2i+1); dims 64..127
    pass through."""
    rng = np.random.Generator(np.random.PCG64(13))
    y = _distinct_row(rng)
    one, zero = np.ones(32, np.float32), np.zeros(32, np.float32)
    assert np.array_equal(oracle.rope_row(y, one, zero, style), y)
    out = oracle.rope_row(y, zero, one, style)
    want = y.copy()
    for i in range(32):
        ia, ib = (i, i + 32) if style == wl.ROPE_NEOX else (2 * i, 2 * i + 1)
        want[ia] = y[ib] ^ 0x8000
        want[ib] = y[ia]
    assert np.array_equal(out, want)


@pytest.mark.parametrize("style", [wl.ROPE_NEOX, wl.ROPE_INTERLEAVED])
def test_rope_single_pair_and_general(style):
    """Only the pair whose table entry is a rotation changes, by that rotation
    (fp64, within one bf16 rounding and fp32 product error); then a general
    table against the fp64 rotation."""
    rng = np.random.Generator(np.random.PCG64(14))
    for i0 in (0, 5, 31):
        y = _distinct_row(rng)
        c = np.ones(32, np.float32)
        s = np.zeros(32, np.float32)
        th = 0.7
        c[i0], s[i0] = np.float32(np.cos(th)), np.float32(np.sin(th))
        out = oracle.rope_row(y, c, s, style)
        ia, ib = (i0, i0 + 32) if style == wl.ROPE_NEOX else (2 * i0, 2 * i0 + 1)
        changed = np.nonzero(out != y)[0]
        assert set(changed.tolist()) <= {ia, ib}
        yf = wl.bf16_bits_to_f32(y).astype(np.float64)
        of = wl.bf16_bits_to_f32(out).astype(np.float64)
        a, b = yf[ia], yf[ib]
        ra = a * float(c[i0]) - b * float(s[i0])
        rb = b * float(c[i0]) + a * float(s[i0])
        tol = lambda r: 2.0 ** -8 * abs(r) + 2.0 ** -22 * (abs(a) + abs(b))
        assert abs(of[ia] - ra) <= tol(ra) and abs(of[ib] - rb) <= tol(rb)
    cos, sin = wl.rope_tables(64)
    for p in (1, 17, 63):
        y = _distinct_row(rng)
        out = wl.bf16_bits_to_f32(oracle.rope_row(y, cos[p], sin[p], style)).astype(np.float64)
        yf = wl.bf16_bits_to_f32(y).astype(np.float64)
        for i in range(32):
            ia, ib = (i, i + 32) if style == wl.ROPE_NEOX else (2 * i, 2 * i + 1)
            a, b = yf[ia], yf[ib]
            ra = a * float(cos[p, i]) - b * float(sin[p, i])
            rb = b * float(cos[p, i]) + a * float(sin[p, i])
            t = 2.0 ** -22 * (abs(a) + abs(b))
            assert abs(out[ia] - ra) <= 2.0 ** -8 * abs(ra) + t
            assert abs(out[ib] - rb) <= 2.0 ** -8 * abs(rb) + t
        assert np.array_equal(out[64:], yf[64:])


# -------------------------------------------------------------- K and Q ops
def test_cache_store_placement_and_skip():
    """Slot s -> page s//64, offset s%64; payload at o*64, exponent word at
    4096 + o*4; a negative slot writes nothing; slot 0 is an ordinary slot;
    every byte not written keeps its sentinel value."""
    rng = np.random.Generator(np.random.PCG64(15))
    T = 4
    k = wl.to_bf16_bits(rng.standard_normal((T, 128)))
    gamma = wl.to_bf16_bits(1 + 0.1 * rng.standard_normal(128))
    pos = np.array([3, 9, 0, 7], np.int64)
    cos, sin = wl.rope_tables(16)
    slots = np.array([5, -1, 0, 64 + 7], np.int64)
    cache0 = rng.integers(0, 256, (2, 4352), dtype=np.uint8)
    cache = cache0.copy()
    st = oracle.k_norm_rope_pack_store(k, gamma, 1e-6, pos, cos, sin, wl.ROPE_NEOX, slots, cache)
    assert st == 0
    touched = np.zeros_like(cache, bool)
    for t in (0, 2, 3):
        y = oracle.rmsnorm_row(k[t], gamma, 1e-6)
        y = oracle.rope_row(y, cos[pos[t]], sin[pos[t]], wl.ROPE_NEOX)
        r = oracle.quant_pack_row(y)
        b, o = divmod(int(slots[t]), 64)
        assert np.array_equal(cache[b, o * 64:o * 64 + 64], r["payload"])
        assert np.array_equal(cache[b, 4096 + 4 * o:4096 + 4 * o + 4], r["exp"])
        touched[b, o * 64:o * 64 + 64] = True
        touched[b, 4096 + 4 * o:4096 + 4 * o + 4] = True
    assert np.array_equal(cache[~touched], cache0[~touched])


def test_out_of_range_rows_are_skipped():
    rng = np.random.Generator(np.random.PCG64(16))
    k = wl.to_bf16_bits(rng.standard_normal((3, 128)))
    gamma = wl.to_bf16_bits(np.ones(128))
    cos, sin = wl.rope_tables(8)
    cache0 = rng.integers(0, 256, (1, 4352), dtype=np.uint8)
    cache = cache0.copy()
    st = oracle.k_norm_rope_pack_store(k, gamma, 1e-6, np.array([8, -1, 2]), cos, sin, 0,
                                       np.array([1, 2, 64]), cache)
    assert st == -1 and np.array_equal(cache, cache0)


def test_golden_midpoint_key_slot():
    w = wl.make("tiny_gamma1")
    cache = w.cache_init.copy()
    oracle.k_norm_rope_pack_store(w.k, w.gamma, w.eps, w.positions, w.cos, w.sin,
                                  w.rope_style, w.slot_mapping, cache)
    pay, exps = golden.midpoint_key_slot()
    b, o = divmod(int(w.slot_mapping[3]), 64)
    assert w.positions[3] == 0
    assert np.array_equal(cache[b, o * 64:o * 64 + 64], pay)
    assert np.array_equal(cache[b, 4096 + 4 * o:4096 + 4 * o + 4], exps)


def test_golden_tiny_query_midpoints():
    """Tiny token 3: head h, group g holds 2^(h-16+g) * {6, +-.25, +-.75,
    +-1.25, +-1.75, +-2.5, +-3.5, +-5, 0...} at position 0; by the grid and
    even ties its payload bytes are 07 20 2a 4a 4c 6c 6e 0e then zeros, and
    its exponent byte is 127+h-16+g."""
    w = wl.make("tiny")
    qf, qs, wt, st = oracle.q_rope_pack_weights(w.q, w.w, w.positions, w.cos, w.sin, w.rope_style)
    assert st == 0
    grp = np.array([0x07, 0x20, 0x2a, 0x4a, 0x4c, 0x6c, 0x6e, 0x0e] + [0] * 8, np.uint8)
    for h in range(w.H):
        assert np.array_equal(qf[3, h], np.tile(grp, 4))
        assert list(qs[3, h]) == [127 + h - 16 + g for g in range(4)]
    # token 1 is all zeros: payload 0, exponents 1
    assert not qf[1].any() and np.all(qs[1] == 1)


def test_weights_closed_form():
    """weights = w * H^-1/2 * D^-1/2 in fp32 (aiter API: plain weight, nothing
    folded; sglang Summary: fp32 head weights): exact w/64 for H=32, the
    correctly rounded product for H=64."""
    rng = np.random.Generator(np.random.PCG64(17))
    for H in (32, 64):
        T = 8
        q = np.zeros((T, H, 128), np.uint16)
        w = wl.to_bf16_bits(rng.standard_normal((T, H)) * 10)
        cos, sin = wl.rope_tables(4)
        _, _, wt, st = oracle.q_rope_pack_weights(q, w, np.zeros(T, np.int64), cos, sin, 0)
        wf = wl.bf16_bits_to_f32(w)
        if H == 32:
            assert np.array_equal(wt, (wf / np.float32(64)).astype(np.float32))
        else:
            getcontext().prec = 60
            s = Decimal(1) / Decimal(H * 128).sqrt()
            want = np.array([float(Decimal(float(v)) * s) for v in wf.ravel()], np.float64)
            assert np.all(ulp_diff_f32(wt.ravel(), want.astype(np.float32)) == 0)


@pytest.mark.floor_reading
def test_oracle_tiny_digest():
    """Drift guard: the oracle's Tiny outputs hash to the committed digest
    written by tests/golden/make_oracle_digest.py (which calls only the
    oracle)."""
    from tests.golden import make_oracle_digest as mod
    assert mod.compute() == mod.read_committed()


def _quarter_turn_tables():
    cos, sin = wl.rope_tables(8)
    cos[5], sin[5] = 0.0, 1.0  # position 5 turns every pair by a quarter
    return cos, sin


def _quarter_turn_row(y, style):
    """(a, b) -> (-b, a) on the 32 RoPE pairs, by index manipulation."""
    out = y.copy()
    for i in range(32):
        ia, ib = (i, i + 32) if style == wl.ROPE_NEOX else (2 * i, 2 * i + 1)
        out[ia] = y[ib] ^ 0x8000
        out[ib] = y[ia]
    return out


@pytest.mark.parametrize("style", [wl.ROPE_NEOX, wl.ROPE_INTERLEAVED])
def test_k_op_closed_form_composition(style):
    """A constant-8 key row normalises to gamma exactly; at a quarter-turn
    position the stored slot must be the packed quarter-turned gamma (the
    steps in the pages' order: RMSNorm, then RoPE, then the quantisers)."""
    rng = np.random.Generator(np.random.PCG64(18))
    gamma = wl.to_bf16_bits(1 + 0.1 * rng.standard_normal(128))
    k = wl.to_bf16_bits(np.full((1, 128), 8.0))
    cos, sin = _quarter_turn_tables()
    cache = np.zeros((1, 4352), np.uint8)
    oracle.k_norm_rope_pack_store(k, gamma, 1e-6, np.array([5]), cos, sin, style,
                                  np.array([3]), cache)
    r = oracle.quant_pack_row(_quarter_turn_row(gamma, style))
    assert np.array_equal(cache[0, 192:256], r["payload"])
    assert np.array_equal(cache[0, 4096 + 12:4096 + 16], r["exp"])


@pytest.mark.parametrize("style", [wl.ROPE_NEOX, wl.ROPE_INTERLEAVED])
def test_q_op_closed_form_composition(style):
    """At a quarter-turn position each query row is packed as its
    quarter-turned self; at position 0 (cos 1, sin 0) as itself."""
    rng = np.random.Generator(np.random.PCG64(19))
    q = wl.to_bf16_bits(rng.standard_normal((2, 3, 128)))
    w = wl.to_bf16_bits(rng.standard_normal((2, 3)))
    cos, sin = _quarter_turn_tables()
    qf, qs, _, st = oracle.q_rope_pack_weights(q, w, np.array([5, 0]), cos, sin, style)
    assert st == 0
    for h in range(3):
        r = oracle.quant_pack_row(_quarter_turn_row(q[0, h], style))
        assert np.array_equal(qf[0, h], r["payload"]) and np.array_equal(qs[0, h], r["exp"])
        r = oracle.quant_pack_row(q[1, h])
        assert np.array_equal(qf[1, h], r["payload"]) and np.array_equal(qs[1, h], r["exp"])

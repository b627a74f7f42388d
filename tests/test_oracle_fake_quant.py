"""Pins of the oracle's torch-shaped fake quantisation ("dsv4.1: RoPE and FP4
packing kernels" (sglang PR 39656), Summary: the RoPE tail plus FP4
fake-quant, per-32 UE8M0 by default and per-16 E4M3 for compressed KV,
keeping the bf16 round trip after RoPE and round half to even).  Checked
against exact rational arithmetic, torch's float8_e4m3fn rounding of the
scale, and closed forms."""
from fractions import Fraction as Fr

import numpy as np
import torch

import oracle
from fp4_sparse_attention_fp4idx_gb300 import workloads as wl
from tests.test_oracle_pins import exact_code, exact_exponent

GRID = [Fr(0), Fr(1, 2), Fr(1), Fr(3, 2), Fr(2), Fr(3), Fr(4), Fr(6)]


def bf16(x) -> np.ndarray:
    return wl.to_bf16_bits(np.asarray(x, np.float32))


def f32(bits) -> np.ndarray:
    return wl.bf16_bits_to_f32(bits)


def e4m3_round(v: float) -> float:
    return float(torch.tensor([v], dtype=torch.float32).to(torch.float8_e4m3fn)
                 .to(torch.float32)[0])


def nearest_e2m1(v: Fr) -> int:
    """Nearest grid code of |v| (saturating at 6), ties to the even code."""
    a = abs(v)
    best = min(range(8), key=lambda m: (abs(GRID[m] - a), m % 2))
    return best


def test_mode0_is_per32_ue8m0_exact():
    """Mode 0: each group's exponent from exact rationals, each value the
    nearest grid value at that scale (ties to even), exactly."""
    rng = np.random.Generator(np.random.PCG64(21))
    for _ in range(60):
        row = bf16(rng.standard_normal(128) * 10.0 ** rng.uniform(-6, 6))
        got = f32(oracle.fake_quant_row(row, 0))
        x = f32(row)
        for g in range(4):
            z = [Fr(float(v)) for v in x[32 * g:32 * g + 32]]
            e = exact_exponent(max(abs(v) for v in z))
            s = Fr(2) ** (e - 127)
            for i, v in enumerate(z):
                m = exact_code(abs(v) / s)
                want = GRID[m] * s * (-1 if (v < 0 and m) else 1)
                assert Fr(float(got[32 * g + i])) == want


def test_mode1_per16_e4m3_exact():
    """Mode 1: s = E4M3(rn32(amax/6)) (torch's rounding), codes the nearest
    E2M1 of rn32(x/s) with ties to even, values code * s exactly."""
    rng = np.random.Generator(np.random.PCG64(22))
    for _ in range(60):
        row = bf16(rng.standard_normal(128) * 10.0 ** rng.uniform(-2, 2.5))
        got = f32(oracle.fake_quant_row(row, 1))
        x = f32(row)
        for g in range(8):
            z = x[16 * g:16 * g + 16]
            amax = np.float32(np.max(np.abs(z)))
            s = e4m3_round(float(np.float32(amax / np.float32(6.0))))
            for i, v in enumerate(z):
                if s == 0.0:
                    assert got[16 * g + i] == 0.0
                    continue
                q = Fr(float(np.float32(v) / np.float32(s)))
                m = nearest_e2m1(q)
                want = GRID[m] * Fr(s) * (-1 if (v < 0 and m) else 1)
                assert Fr(float(got[16 * g + i])) == want


def test_mode1_midpoints_closed_form():
    """A group with amax 6 has scale 1; the E2M1 midpoints 0.25, 0.75, 1.25,
    1.75, 2.5, 3.5, 5 go to the even codes 0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0."""
    z = np.zeros(16, np.float32)
    z[0] = 6.0
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    want = [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]
    z[1:8] = mids
    z[8:15] = [-m for m in mids]
    row = np.zeros(128, np.float32)
    row[:16] = z
    got = f32(oracle.fake_quant_row(bf16(row), 1))
    assert got[0] == 6.0
    assert list(got[1:8]) == want
    assert list(got[8:15]) == [-w if w else 0.0 for w in want]
    assert not np.any(np.signbit(got[8:9]))  # -0.25 -> +0 (no negative zero)


def test_mode1_tiny_group_is_zero_and_saturation():
    """amax/6 below half the smallest E4M3 subnormal rounds the scale to 0:
    the group is all zeros.  amax/6 above 448 saturates the scale at 448 and
    the codes at 6: values clip at +-2688."""
    row = np.zeros(128, np.float32)
    row[:16] = 1e-4
    row[16:32] = np.linspace(-1e4, 1e4, 16)
    got = f32(oracle.fake_quant_row(bf16(row), 1))
    assert np.all(got[:16] == 0.0)
    assert got[16] == -2688.0 and got[31] == 2688.0


def test_rope_then_fake_quant_at_position_zero():
    """At position 0 RoPE is the identity, so the call equals the row-level
    fake quantisation; rows take their token's position."""
    cos, sin = wl.rope_tables(8)
    rng = np.random.Generator(np.random.PCG64(23))
    x = bf16(rng.standard_normal((6, 128)))
    for mode in (0, 1):
        out, st = oracle.rope_fake_quant(x, 3, np.array([0, 5], np.int64), cos, sin, 0, mode)
        assert st == 0
        for r in range(3):
            assert np.array_equal(out[r], oracle.fake_quant_row(x[r], mode))
        moved = [not np.array_equal(out[r], oracle.fake_quant_row(x[r], mode)) for r in (3, 4, 5)]
        assert all(moved)

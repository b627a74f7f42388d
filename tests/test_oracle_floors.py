"""The scale floors of the two quantisation stages: what the pages fix, what
they leave open, and which bytes hang on the reading taken.

"dsv4.1: RoPE and FP4 packing kernels" (sglang PR 39656), review: the
indexer packer (stage 2) keeps amax / 6.0f and a floor applied after the
division, and the packer "has a different scale floor from fake_quant_fp4"
(stage 1).  "DeepSeek-V4 FP4: fused_compress FP4 scatter +
rmsnorm_rope_rotate FP4 KV-cache kernel" (aiter PR 4029), review: the FP4
quantiser's amax has an all-zero-group eps floor.  No floor value is printed.

The oracle floors the stage-1 amax before the division and the stage-2
quotient after it, both at 2^-126.  These tests show (against exact
rational arithmetic, not the oracle's own formula) that every floor pair in
(0, 6*2^-126] x (0, 2^-126] gives the same exponent for every group, that a
larger floor changes exactly the groups below it, and which groups of the
shipped workloads are decided by the floor at all.
"""
from fractions import Fraction as Fr

import numpy as np
import pytest

import oracle
from fp4_sparse_attention_fp4idx_gb300 import workloads as wl
from tests.test_oracle_pins import (all_finite_bf16, bf16_value, exact_code,
                                    exact_exponent, GRID)

TINY = 2.0 ** -126
# (stage-1 amax floor, stage-2 quotient floor) pairs that the pages allow and
# that all keep the exponent clamp's lower bound unreachable
FAMILY = [(TINY, TINY), (2.0 ** -149, 2.0 ** -149), (6 * TINY, TINY), (TINY / 6, 2.0 ** -140),
          (2.0 ** -130, 2.0 ** -127), (TINY, 0.0), (0.0, TINY)]


def positive_bf16_amax():
    b = all_finite_bf16()
    return [bf16_value(int(x)) for x in b if not (int(x) >> 15)]


def exponent_with_floors(a: float, amax_floor: float, quot_floor: float) -> int:
    """The group exponent by exact rational arithmetic: A = max(a, amax
    floor); t = A/6 rounded to fp32; e = biased exponent of ceil_pow2(max(t,
    quotient floor)), at least 1."""
    A = max(Fr(a), Fr(amax_floor))
    t = Fr(float(np.float32(A / 6))) if A else Fr(0)
    t = max(t, Fr(quot_floor))
    if t == 0:
        return 1
    return exact_exponent(6 * t)


def test_floor_family_gives_one_exponent_for_every_bf16_amax():
    """For every non-negative finite bf16 amax, every floor pair of the family
    gives the exponent of the reading taken, which is the exact
    ceil_pow2(amax/6) exponent (at least 1)."""
    z = np.zeros(32, np.float32)
    for a in positive_bf16_amax():
        z[0] = a
        want = exact_exponent(Fr(a))
        for af, qf in FAMILY:
            _, e = oracle.quant_group_floors(z, af, qf)
            assert e == want, (a, af, qf, e, want)


@pytest.mark.parametrize("floor", [2.0 ** -100, 1e-4 / 6, 2.0 ** -3])
def test_larger_floor_changes_exactly_the_groups_below_it(floor):
    """A floor above the family (as a quotient floor F, or as an amax floor
    6F) changes a group's exponent exactly when its amax is below 6F, and
    then gives the floor's own exponent."""
    z = np.zeros(32, np.float32)
    eF = exponent_with_floors(0.0, 0.0, floor)
    for a in positive_bf16_amax()[::7]:
        z[0] = a
        base = exact_exponent(Fr(a))
        for af, qf in ((0.0, floor), (6 * floor, 0.0)):
            _, e = oracle.quant_group_floors(z, af, qf)
            assert e == exponent_with_floors(a, af, qf)
            if base >= eF:
                assert e == base
            else:
                assert e == eF and Fr(a) < 6 * Fr(floor)


def two_stage_exact(row_bits):
    """Both stages of one row by exact rationals (the pages' order: stage 1
    fake-quantises and dequantises, stage 2 packs): (payload, exponents)."""
    vals = [Fr(bf16_value(int(b))) for b in row_bits]
    pay = np.zeros(64, np.uint8)
    exps = np.zeros(4, np.uint8)
    nib = np.zeros(128, np.uint8)
    for g in range(4):
        z = vals[32 * g:32 * g + 32]
        e1 = exact_exponent(max(abs(x) for x in z))
        s1 = Fr(2) ** (e1 - 127)
        u = [GRID[exact_code(abs(x) / s1)] * s1 * (-1 if x < 0 else 1) for x in z]
        e2 = exact_exponent(max(abs(x) for x in u))
        s2 = Fr(2) ** (e2 - 127)
        for i, x in enumerate(u):
            m = exact_code(abs(x) / s2)
            nib[32 * g + i] = m | (8 if (x < 0 and m) else 0)
        exps[g] = e2
    pay[:] = nib[0::2] | (nib[1::2] << 4)
    return pay, exps


def test_tiny_groups_two_stage_exact():
    """Rows at the bottom of the range -- bf16 subnormals, the smallest
    normals and values around 6*2^-126 -- through both stages, against exact
    rational arithmetic.  The bytes of these groups are the ones a floor
    reading could touch."""
    rng = np.random.Generator(np.random.PCG64(81))
    for it in range(60):
        kind = it % 3
        if kind == 0:
            row = wl.subnormal_bf16(rng, 128)
        elif kind == 1:
            row = wl.to_bf16_bits(rng.standard_normal(128) * 2.0 ** rng.integers(-130, -115))
        else:
            row = wl.to_bf16_bits(rng.uniform(-6, 6, 128) * 2.0 ** -126)
        pay, exps = two_stage_exact(row)
        r = oracle.quant_pack_row(row)
        assert np.array_equal(r["payload"], pay), it
        assert np.array_equal(r["exp"], exps), it
        for af, qf in FAMILY:
            rf = oracle.quant_pack_row_floors(row, af, 0.0, 0.0, qf)
            assert np.array_equal(rf["payload"], pay) and np.array_equal(rf["exp"], exps)


def stored_exponents(w):
    cache = w.cache_init.copy()
    oracle.k_norm_rope_pack_store(w.k, w.gamma, w.eps, w.positions, w.cos, w.sin,
                                  w.rope_style, w.slot_mapping, cache)
    _, qs, _, _ = oracle.q_rope_pack_weights(w.q, w.w, w.positions, w.cos, w.sin, w.rope_style)
    ok = w.slot_mapping >= 0
    b, o = w.slot_mapping[ok] // 64, w.slot_mapping[ok] % 64
    kexp = np.stack([cache[b, 4096 + 4 * o + g] for g in range(4)], 1)
    return np.nonzero(ok)[0], kexp, qs.reshape(w.T, w.H, 4)


@pytest.mark.parametrize("name", ["tiny", "tiny_gamma1", "decode", "prefill", "mtp"])
def test_floor_decided_groups_of_the_workloads(name):
    """The groups whose bytes a floor reading decides.  Exponent byte 1 is
    the floor's exponent: in the shipped workloads only the Tiny config has
    such groups -- its all-zero token 1 (key and every query head) and its
    subnormal token 2 (every query head; the key row is rescaled by RMSNorm).
    Every other group sits far above the floor (exponent byte >= 9, and >=
    111 outside Tiny's keys), so a real floor below 2^-118 (below 2^-17 for
    the non-Tiny configs) would change no byte outside those rows."""
    w = wl.make(name)
    with oracle.threads():
        toks, kexp, qexp = stored_exponents(w)
    kfloor = sorted(set(toks[np.any(kexp == 1, 1)].tolist()))
    qfloor = sorted(set(np.nonzero(np.any(qexp == 1, (1, 2)))[0].tolist()))
    if name.startswith("tiny"):
        assert kfloor == [1] and qfloor == [1, 2]
        assert np.all(kexp[toks == 1] == 1) and np.all(qexp[[1, 2]] == 1)
        assert kexp[kexp > 1].min() >= 9 and qexp[qexp > 1].min() >= 111
    else:
        assert kfloor == [] and qfloor == []
        assert min(kexp.min(), qexp.min()) >= 111


def test_threaded_oracle_is_identical():
    """The token loops on all host cores give the single-threaded bytes,
    including the last-writer rule for a slot written twice."""
    w = wl.make("decode")
    w.slot_mapping[7] = w.slot_mapping[3] if w.slot_mapping[3] >= 0 else w.slot_mapping[4]
    outs = []
    for n in (1, oracle.threads_available()):
        with oracle.threads(n):
            cache = w.cache_init.copy()
            oracle.k_norm_rope_pack_store(w.k, w.gamma, w.eps, w.positions, w.cos, w.sin,
                                          w.rope_style, w.slot_mapping, cache)
            qf, qs, wt, _ = oracle.q_rope_pack_weights(w.q, w.w, w.positions, w.cos, w.sin,
                                                       w.rope_style)
            outs.append((cache, qf, qs, wt))
    for a, b in zip(*outs):
        assert np.array_equal(a, b)

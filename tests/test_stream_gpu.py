"""GPU parity of the streaming pre-pass kernel (64-row work units fed by a
producer warp, four lanes per row): the path taken for both output modes
(FP4 and FP8), with or without the 128-point rotation, when the head count
is a multiple of 16, and for every key-only call.  The cases leave ragged units and slices, use every
query-row layout the producer copies (contiguous rows, contiguous heads
under a larger token stride, one copy per row), put the quantiser's edge
rows at both row parities of a quarter-warp, and feed out-of-range
positions.  Bytes must equal the oracle's; weights within 1 ulp."""
import numpy as np
import pytest
import torch

from fp4_sparse_attention_fp4idx_gb300 import workloads as wl
from tests.gpu_util import (DeviceWorkload, F, assert_bytes_equal, assert_same, assert_weights,
                            run_oracle)
from tests.test_fp8_gpu import assert_fp8_same, run_gpu as run_fp8, run_ref as run_fp8_ref

pytestmark = pytest.mark.gpu

STYLES = [wl.ROPE_NEOX, wl.ROPE_INTERLEAVED]


@pytest.mark.parametrize("hadamard", [False, True], ids=["plain", "rotated"])
@pytest.mark.parametrize("style", STYLES)
@pytest.mark.parametrize("T,H", [(1, 16), (3, 16), (5, 48), (63, 32), (64, 16), (65, 64),
                                 (130, 128), (301, 32)])
def test_stream_ragged(T, H, style, hadamard):
    """Units that end mid-slice (T*H not a multiple of 64), key units that
    end mid-unit (T not a multiple of 64), one token, 128 heads."""
    w = wl.make_random(T, H, style, seed=2000 + 13 * T + H)
    ref = run_oracle(w, hadamard=hadamard)
    for mode in ("fused", "separate"):
        d = DeviceWorkload(w)
        assert_same(w, d.run(mode, hadamard=hadamard), ref)
        assert int(d.err.item()) == 0


@pytest.mark.parametrize("T", [9578, 9579])
def test_stream_ring_depth_boundary(T):
    """The ring is 8 stages deep while the largest producer share of a
    launch is at most 16 units, else 12.  At 64 heads on 152 SMs the fused
    launch crosses that line between T = 9578 (150 key + 9578 query units:
    64 per CTA, shares of 16) and T = 9579 (9729 units: 65 per CTA, a share
    of 17); both depths wrap their ring many times and must give the same
    bytes as the oracle."""
    w = wl.make_random(T, 64, wl.ROPE_NEOX, seed=2500 + T)
    ref = run_oracle(w)
    d = DeviceWorkload(w)
    assert_same(w, d.run("fused"), ref)
    assert int(d.err.item()) == 0


@pytest.mark.parametrize("hadamard", [False, True], ids=["plain", "rotated"])
@pytest.mark.parametrize("style", STYLES)
@pytest.mark.parametrize("scale", [1.0, 40.0, 1e-3, 3e4])
@pytest.mark.floor_reading
def test_stream_special_rows(style, scale, hadamard):
    """All-zero, subnormal and exact-midpoint query rows on even and odd rows
    of a unit (the two part orders), with the keys of the same tokens."""
    w = wl.make_random(70, 16, style, seed=int(scale * 7) + 31 * style + 5, scales=(scale,))
    rng = np.random.Generator(np.random.PCG64(17 + style))
    w.q[0] = 0
    w.k[0] = 0
    w.q[1] = wl.subnormal_bf16(rng, 16 * 128).reshape(16, 128)
    w.k[1] = wl.subnormal_bf16(rng, 128)
    for t in (2, 3):
        for h in range(16):
            w.q[t, h] = wl.to_bf16_bits(np.concatenate(
                [wl.midpoint_group_values(h - 8 + g + t) for g in range(4)]))
        w.positions[t] = 0
    w.k[4] = wl.to_bf16_bits(wl.midpoint_key_row())
    d = DeviceWorkload(w)
    assert_same(w, d.run("fused", hadamard=hadamard), run_oracle(w, hadamard=hadamard))
    assert int(d.err.item()) == 0


@pytest.mark.parametrize("style", STYLES)
def test_stream_query_layouts(style):
    """The producer's three ways of copying query rows: one copy per unit
    (dense), one per 16-row slice (heads contiguous, token stride larger than
    H*128), one per row (head stride 256); keys with a row stride too."""
    w = wl.make_random(50, 32, style, seed=88 + style)
    d = DeviceWorkload(w)
    f = F()
    rc, rqf, rqs, rwt = run_oracle(w)
    big1 = torch.zeros((50, 40, 128), dtype=torch.bfloat16, device="cuda")
    big1[:, 3:35] = d.q
    big2 = torch.zeros((50, 64, 128), dtype=torch.bfloat16, device="cuda")
    big2[:, ::2] = d.q
    bigk = torch.zeros((50, 2, 128), dtype=torch.bfloat16, device="cuda")
    bigk[:, 1] = d.k
    kv = bigk[:, 1]
    for qv in (d.q, big1[:, 3:35], big2[:, ::2]):
        qf, qs, wt = f.q_rope_pack_weights(qv, d.wt, d.pos, d.cos, d.sin,
                                           rope_style=w.rope_style)
        torch.cuda.synchronize()
        assert_bytes_equal(qf.cpu().numpy(), rqf, f"q_fp4 strides {qv.stride()}")
        assert_bytes_equal(qs.cpu().numpy(), rqs, f"q_scale strides {qv.stride()}")
        assert_weights(wt.cpu().numpy(), rwt)
        d.reset_cache()
        qf, qs, wt = f.indexer_prepass(kv, d.gamma, d.slots, d.cache, qv, d.wt, d.pos, d.cos,
                                       d.sin, eps=w.eps, rope_style=w.rope_style)
        torch.cuda.synchronize()
        assert_same(w, (d.cache.cpu().numpy(), qf.cpu().numpy(), qs.cpu().numpy(),
                        wt.cpu().numpy()), (rc, rqf, rqs, rwt))


def test_stream_out_of_range_positions():
    """A query token whose position is outside [0, max_pos) is skipped as a
    whole (its slices are flagged, nothing of it is written); the key rows
    of such tokens are skipped and flagged; the rest is exact."""
    w = wl.make_random(40, 32, wl.ROPE_INTERLEAVED, seed=23, max_pos=100)
    w.positions[3] = 100
    w.positions[17] = -1
    w.positions[39] = 1 << 40
    for mode in ("fused", "separate"):
        d = DeviceWorkload(w)
        sentinel = torch.full((40, 32, 64), 0xA5, dtype=torch.uint8, device="cuda")
        d.reset_cache()
        if mode == "fused":
            qf, qs, wt = F().indexer_prepass(d.k, d.gamma, d.slots, d.cache, d.q, d.wt, d.pos,
                                             d.cos, d.sin, eps=w.eps, rope_style=w.rope_style,
                                             q_fp4=sentinel, err_flags=d.err)
        else:
            F().k_norm_rope_pack_store(d.k, d.gamma, d.pos, d.cos, d.sin, d.slots, d.cache,
                                       eps=w.eps, rope_style=w.rope_style, err_flags=d.err)
            qf, qs, wt = F().q_rope_pack_weights(d.q, d.wt, d.pos, d.cos, d.sin,
                                                 rope_style=w.rope_style, q_fp4=sentinel,
                                                 err_flags=d.err)
        torch.cuda.synchronize()
        assert int(d.err.item()) & F().ERRFLAG_POSITION
        rc, rqf, rqs, rwt = run_oracle(w)
        assert_bytes_equal(d.cache.cpu().numpy(), rc, "cache")
        good = np.setdiff1d(np.arange(40), [3, 17, 39])
        qfn = qf.cpu().numpy()
        assert_bytes_equal(qfn[good], rqf[good], "q_fp4")
        assert_bytes_equal(qs.cpu().numpy()[good], rqs[good], "q_scale")
        assert_weights(wt.cpu().numpy()[good], rwt[good])
        assert np.all(qfn[[3, 17, 39]] == 0xA5)


@pytest.mark.parametrize("hadamard", [False, True], ids=["plain", "rotated"])
def test_stream_repeat_and_reuse(hadamard):
    """Two launches in a row on the prefill workload give the same bytes (no
    state carried between launches)."""
    w = wl.make("prefill")
    d = DeviceWorkload(w)
    a = d.run("fused", hadamard=hadamard)
    b = d.run("fused", hadamard=hadamard)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    assert int(d.err.item()) == 0


@pytest.mark.parametrize("hadamard", [False, True], ids=["plain", "rotated"])
@pytest.mark.parametrize("style", STYLES)
@pytest.mark.parametrize("T,H", [(1, 16), (5, 48), (63, 32), (65, 64), (130, 128), (301, 32)])
def test_stream_fp8_ragged(T, H, style, hadamard):
    """The FP8 output mode: 8448-byte cache pages and 128-byte query code
    rows byte for byte, the weights (row scale folded in) within 1 ulp, on
    ragged units and slices, with and without the rotation."""
    w = wl.make_random(T, H, style, seed=3000 + 13 * T + H)
    ref = run_fp8_ref(w, hadamard=hadamard)
    for mode in ("fused", "separate"):
        d = DeviceWorkload(w)
        assert_fp8_same(f"T={T} H={H} {mode}", run_fp8(d, mode, hadamard=hadamard), ref)
        assert int(d.err.item()) == 0


@pytest.mark.parametrize("style", STYLES)
@pytest.mark.parametrize("scale", [1.0, 1e-3, 3e4])
@pytest.mark.floor_reading
def test_stream_fp8_special_rows(style, scale):
    """FP8 rows at the scale's edges on both row parities: all-zero and
    subnormal rows (the 2^-126 floor), and query rows whose amax/448 is an
    exact power of two (no rounding up of the scale), at position 0."""
    w = wl.make_random(70, 16, style, seed=int(scale * 11) + 31 * style + 9, scales=(scale,))
    rng = np.random.Generator(np.random.PCG64(29 + style))
    w.q[0] = 0
    w.k[0] = 0
    w.q[1] = wl.subnormal_bf16(rng, 16 * 128).reshape(16, 128)
    w.k[1] = wl.subnormal_bf16(rng, 128)
    for t in (2, 3):
        for h in range(16):
            top = 448.0 * 2.0 ** (h - 8)
            row = rng.uniform(-0.9, 0.9, 128) * top
            row[(7 * h + t) % 128] = top if h % 2 else -top
            w.q[t, h] = wl.to_bf16_bits(row)
        w.positions[t] = 0
    d = DeviceWorkload(w)
    assert_fp8_same("special rows", run_fp8(d, "fused"), run_fp8_ref(w))
    assert int(d.err.item()) == 0


def test_stream_fp8_query_layouts():
    """The FP8 mode under the producer's three query-row copy layouts (one
    copy per unit, per 16-row slice, per row) and a key row stride of 256."""
    w = wl.make_random(50, 32, wl.ROPE_NEOX, seed=90)
    d = DeviceWorkload(w)
    f = F()
    rc, rq, rw = run_fp8_ref(w)
    big1 = torch.zeros((50, 40, 128), dtype=torch.bfloat16, device="cuda")
    big1[:, 3:35] = d.q
    big2 = torch.zeros((50, 64, 128), dtype=torch.bfloat16, device="cuda")
    big2[:, ::2] = d.q
    bigk = torch.zeros((50, 2, 128), dtype=torch.bfloat16, device="cuda")
    bigk[:, 1] = d.k
    for qv in (d.q, big1[:, 3:35], big2[:, ::2]):
        cache = torch.from_numpy(wl.fp8_sentinel_cache(w)).cuda()
        qo, wt = f.indexer_prepass_fp8(bigk[:, 1], d.gamma, d.slots, cache, qv, d.wt, d.pos,
                                       d.cos, d.sin, eps=w.eps, rope_style=w.rope_style)
        torch.cuda.synchronize()
        assert_fp8_same(f"strides {qv.stride()}", (cache.cpu().numpy(), qo.cpu().numpy(),
                                                   wt.cpu().numpy()), (rc, rq, rw))


def test_stream_fp8_out_of_range_positions():
    """FP8 mode: a query token whose position is out of range is skipped
    whole and flagged; its key row is skipped and flagged; the rest is exact."""
    w = wl.make_random(40, 32, wl.ROPE_INTERLEAVED, seed=24, max_pos=100)
    w.positions[5] = 100
    w.positions[30] = -3
    d = DeviceWorkload(w)
    cache = torch.from_numpy(wl.fp8_sentinel_cache(w)).cuda()
    sentinel = torch.full((40, 32, 128), 0xA5, dtype=torch.uint8, device="cuda")
    qo, wt = F().indexer_prepass_fp8(d.k, d.gamma, d.slots, cache, d.q, d.wt, d.pos, d.cos,
                                     d.sin, eps=w.eps, rope_style=w.rope_style, q_out=sentinel,
                                     err_flags=d.err)
    torch.cuda.synchronize()
    assert int(d.err.item()) & F().ERRFLAG_POSITION
    rc, rq, rw = run_fp8_ref(w)
    assert_bytes_equal(cache.cpu().numpy(), rc, "fp8 cache")
    good = np.setdiff1d(np.arange(40), [5, 30])
    qn = qo.cpu().numpy()
    assert_bytes_equal(qn[good], rq[good], "fp8 q codes")
    assert_weights(wt.cpu().numpy()[good], rw[good])
    assert np.all(qn[[5, 30]] == 0xA5)

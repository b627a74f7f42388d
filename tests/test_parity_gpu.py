"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.  Bytes (q_fp4, q_scale, the whole paged cache including
the untouched bytes of skipped slots) must match exactly; fp32 head weights
within 1 ulp."""
import numpy as np
import pytest
import torch

import oracle
from fp4_sparse_attention_fp4idx_gb300 import workloads as wl
from tests import golden
from tests.gpu_util import (DeviceWorkload, F, assert_bytes_equal, assert_same,
                            assert_weights, bf16_dev, dev, run_oracle)

pytestmark = pytest.mark.gpu

MODES = ["fused", "separate"]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("name", [pytest.param("tiny", marks=pytest.mark.floor_reading),
                                  pytest.param("tiny_gamma1", marks=pytest.mark.floor_reading),
                                  "decode", "mtp", "prefill"])
def test_config_parity(name, mode):
    w = wl.make(name)
    dw = DeviceWorkload(w)
    gpu = dw.run(mode)
    assert_same(w, gpu, run_oracle(w))
    assert int(dw.err.item()) == 0


def test_large_prefill_parity_full():
    """Full-size large prefill (T=65536, H=64) in the bench's launch
    configuration (one fused launch): the whole cache and every query output
    of all 65,536 tokens against the oracle (run on all host cores)."""
    w = wl.make("large_prefill")
    dw = DeviceWorkload(w)
    gpu = dw.run("fused")
    with oracle.threads():
        ref = run_oracle(w)
    assert_same(w, gpu, ref)


def test_golden_fixtures_on_gpu():
    """The hand-derived slots of the midpoint rows (not oracle output)."""
    w = wl.make("tiny_gamma1")
    cache, qf, qs, _ = DeviceWorkload(w).run("fused")
    pay, exps = golden.midpoint_key_slot()
    b, o = divmod(int(w.slot_mapping[3]), 64)
    assert np.array_equal(cache[b, o * 64:o * 64 + 64], pay)
    assert np.array_equal(cache[b, 4096 + 4 * o:4096 + 4 * o + 4], exps)
    grp = np.array([0x07, 0x20, 0x2a, 0x4a, 0x4c, 0x6c, 0x6e, 0x0e] + [0] * 8, np.uint8)
    for h in range(w.H):
        assert np.array_equal(qf[3, h], np.tile(grp, 4))
        assert list(qs[3, h]) == [127 + h - 16 + g for g in range(4)]


def _rows_to_workload(rows: np.ndarray, H: int, style=wl.ROPE_NEOX) -> wl.Workload:
    """Query/key rows (bf16 bits, [N,128]) at position 0 (RoPE = identity)."""
    n = rows.shape[0]
    T = -(-n // H)
    pad = T * H - n
    q = np.concatenate([rows, np.zeros((pad, 128), np.uint16)]).reshape(T, H, 128)
    cos, sin = wl.rope_tables(4)
    k = q[:, 0, :].copy()
    return wl.Workload("rows", T, H, style, q, np.zeros((T, H), np.uint16), k,
                       wl.to_bf16_bits(np.ones(128)), 1e-6, np.zeros(T, np.int64), cos, sin,
                       np.arange(T, dtype=np.int64), -(-T // 64),
                       np.zeros((-(-T // 64), 4352), np.uint8))


def test_exhaustive_bf16_quantizer_on_gpu():
    """Every finite bf16 value (1) as the amax of its own group and (2) inside
    groups anchored at 6*2^j for every j, through the query path at position
    0 (cos 1, sin 0 makes RoPE the identity exactly), against the oracle."""
    b = np.arange(1 << 16, dtype=np.uint32)
    allv = b[((b >> 7) & 0xFF) != 0xFF].astype(np.uint16)
    vals = (allv.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    mag = np.abs(vals)
    # A group amax above 6*2^125 makes the stage-1 dequantised value overflow
    # (outside the finite domain; see test_domain_boundary_top_binade).
    own = allv[mag <= 6.0 * 2.0 ** 125]
    own = np.concatenate([own, np.zeros((-own.size) % 4, np.uint16)])
    g = np.zeros((own.size, 32), np.uint16)
    g[:, 5] = own
    rows = [g.reshape(-1, 128)]
    groups = []
    for j in range(-126, 126):
        sel = allv[(mag <= 6.0 * 2.0 ** j) & (mag >= 2.0 ** (j - 4))]
        pad = (-sel.size) % 31
        zs = np.concatenate([sel, np.zeros(pad, np.uint16)]).reshape(-1, 31)
        anchor = wl.to_bf16_bits(np.array([6.0 * 2.0 ** j]))[0]
        groups.append(np.concatenate([np.full((zs.shape[0], 1), anchor, np.uint16), zs], 1))
    gg = np.concatenate(groups)
    gg = np.concatenate([gg, np.zeros(((-gg.shape[0]) % 4, 32), np.uint16)])
    rows.append(gg.reshape(-1, 128))
    allrows = np.concatenate(rows)
    w = _rows_to_workload(allrows, 64)
    _, qf, qs, _ = DeviceWorkload(w).run("separate")
    _, rqf, rqs, _ = run_oracle(w)
    assert_bytes_equal(qf, rqf, "exhaustive q_fp4")
    assert_bytes_equal(qs, rqs, "exhaustive q_scale")


@pytest.mark.parametrize("style", [wl.ROPE_NEOX, wl.ROPE_INTERLEAVED])
@pytest.mark.parametrize("T,H", [(1, 1), (5, 3), (64, 16), (300, 17), (7, 33), (3, 65),
                                 (9, 130), (33, 64), (8, 32), (32, 64)])
def test_ragged_shapes(T, H, style):
    """Head counts that do not fill the 16-engine x 4-row batches, single
    tokens, and token counts that leave ragged tails for the key groups."""
    w = wl.make_random(T, H, style, seed=1000 + T * 7 + H)
    for mode in MODES:
        assert_same(w, DeviceWorkload(w).run(mode), run_oracle(w))


@pytest.mark.parametrize("style", [wl.ROPE_NEOX, wl.ROPE_INTERLEAVED])
@pytest.mark.parametrize("rows", [1, 5, 64, 300])
@pytest.mark.parametrize("scale", [1.0, 40.0, 1e-3])
@pytest.mark.floor_reading
def test_row_scale_grid(rows, scale, style):
    """Rows x input scales with an all-zero row, a subnormal row and an exact
    half-way row mixed in (the byte-comparison grid of the sglang PR's
    Verification section)."""
    w = wl.make_random(rows, 8, style, seed=int(rows * 10 + scale * 3) + style,
                       scales=(scale,))
    rng = np.random.Generator(np.random.PCG64(rows))
    if rows >= 3:
        w.q[0] = 0
        w.k[0] = 0
        w.q[1] = wl.subnormal_bf16(rng, 8 * 128).reshape(8, 128)
        w.k[1] = wl.subnormal_bf16(rng, 128)
        for h in range(8):
            w.q[2, h] = wl.to_bf16_bits(np.concatenate(
                [wl.midpoint_group_values(h - 4 + g) for g in range(4)]))
        w.positions[2] = 0
    assert_same(w, DeviceWorkload(w).run("fused"), run_oracle(w))


def test_strided_inputs():
    """q, k and w taken as views with token/head strides larger than dense."""
    w = wl.make_random(40, 12, wl.ROPE_NEOX, seed=77)
    d = DeviceWorkload(w)
    f = F()
    big_q = torch.zeros((40, 24, 128), dtype=torch.bfloat16, device="cuda")
    big_q[:, ::2] = d.q
    qv = big_q[:, ::2]
    big_k = torch.zeros((40, 3, 128), dtype=torch.bfloat16, device="cuda")
    big_k[:, 1] = d.k
    kv = big_k[:, 1]
    big_w = torch.zeros((40, 20), dtype=torch.bfloat16, device="cuda")
    big_w[:, :12] = d.wt
    wv = big_w[:, :12]
    assert qv.stride() == (24 * 128, 256, 1) and kv.stride() == (384, 1) and wv.stride() == (20, 1)
    d.reset_cache()
    f.k_norm_rope_pack_store(kv, d.gamma, d.pos, d.cos, d.sin, d.slots, d.cache, eps=w.eps,
                             rope_style=w.rope_style)
    qf, qs, wt = f.q_rope_pack_weights(qv, wv, d.pos, d.cos, d.sin, rope_style=w.rope_style)
    torch.cuda.synchronize()
    assert_same(w, (d.cache.cpu().numpy(), qf.cpu().numpy(), qs.cpu().numpy(), wt.cpu().numpy()),
                run_oracle(w))


def test_empty_batch_is_a_no_op():
    w = wl.make_random(4, 8, wl.ROPE_NEOX, seed=5)
    d = DeviceWorkload(w)
    f = F()
    e = slice(0, 0)
    before = d.cache.clone()
    qf, qs, wt = f.indexer_prepass(d.k[e], d.gamma, d.slots[e], d.cache, d.q[e], d.wt[e],
                                   d.pos[e], d.cos, d.sin)
    f.k_norm_rope_pack_store(d.k[e], d.gamma, d.pos[e], d.cos, d.sin, d.slots[e], d.cache)
    torch.cuda.synchronize()
    assert qf.shape == (0, 8, 64) and torch.equal(before, d.cache)


def test_out_of_range_rows_are_skipped_and_flagged():
    """A position outside [0, max_pos) or a slot past the cache is skipped
    without any out-of-bounds access and reported in err_flags; the other
    rows are exact."""
    w = wl.make_random(50, 8, wl.ROPE_INTERLEAVED, seed=21, max_pos=100)
    w.positions[3] = 100          # == max_pos
    w.positions[7] = -5
    last = w.num_blocks * 64 - 1
    w.slot_mapping[np.isin(w.slot_mapping, [0, last])] = -1  # keep slots distinct
    w.slot_mapping[11] = w.num_blocks * 64  # one past the last slot: flagged
    w.slot_mapping[12] = last               # the last slot: valid
    w.slot_mapping[13] = 0                  # slot 0: an ordinary slot
    for mode in MODES:
        d = DeviceWorkload(w)
        cache, qf, qs, wt = d.run(mode)
        flags = int(d.err.item())
        assert flags == (F().ERRFLAG_POSITION | F().ERRFLAG_SLOT), flags
        rc, rqf, rqs, rwt = run_oracle(w)
        assert_bytes_equal(cache, rc, "cache")
        good = np.setdiff1d(np.arange(50), [3, 7])
        assert_bytes_equal(qf[good], rqf[good], "q_fp4")
        assert_bytes_equal(qs[good], rqs[good], "q_scale")
        assert_weights(wt[good], rwt[good])


def test_repeatable_and_stream_ordered():
    """Two launches on a side stream give identical bytes."""
    w = wl.make("decode")
    d = DeviceWorkload(w)
    s = torch.cuda.Stream()
    outs = []
    for _ in range(2):
        with torch.cuda.stream(s):
            d.reset_cache()
            qf, qs, wt = F().indexer_prepass(d.k, d.gamma, d.slots, d.cache, d.q, d.wt, d.pos,
                                             d.cos, d.sin, rope_style=w.rope_style)
        s.synchronize()
        outs.append((d.cache.cpu().numpy(), qf.cpu().numpy(), qs.cpu().numpy(), wt.cpu().numpy()))
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a, b)
    assert_same(w, outs[0], run_oracle(w))


def test_host_checks_enqueue_nothing():
    """Bad arguments return a status before any launch (checked on device
    memory here; the CPU suite checks the same codes without a GPU)."""
    f = F()
    w = wl.make_random(4, 8, wl.ROPE_NEOX, seed=6)
    d = DeviceWorkload(w)
    with pytest.raises(f.Fp4idxError) as ei:
        f.k_norm_rope_pack_store(d.k, d.gamma, d.pos, d.cos, d.sin, d.slots, d.cache, eps=0.0)
    assert ei.value.status == f.ERR_ARG
    mis = torch.zeros(4 * 128 + 4, dtype=torch.bfloat16, device="cuda")[4:].view(4, 128)
    with pytest.raises(f.Fp4idxError) as ei:
        f.k_norm_rope_pack_store(mis, d.gamma, d.pos, d.cos, d.sin, d.slots, d.cache)
    assert ei.value.status == f.ERR_ALIGN

"""GPU parity of the torch-shaped RoPE + FP4 fake quantisation
(fp4idx_rope_fake_quant) against the oracle on the same seeded inputs: every
output bf16 bit pattern equal.  Source: "dsv4.1: RoPE and FP4 packing
kernels" (sglang PR 39656), Summary (per-32 UE8M0 by default, per-16 E4M3
for compressed KV, bf16 round trip after RoPE, round half to even)."""
import numpy as np
import pytest
import torch

import oracle
from fp4_sparse_attention_fp4idx_gb300 import workloads as wl
from tests.gpu_util import F, assert_bytes_equal, bf16_dev, dev

pytestmark = pytest.mark.gpu

MODES = [0, 1]


def run_both(x_bits, positions, cos, sin, style, mode, rows_per_token):
    x = bf16_dev(x_bits)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = F().rope_fake_quant(x, dev(positions), dev(cos), dev(sin), rope_style=style,
                              scale_mode=mode, err_flags=err)
    torch.cuda.synchronize()
    got = got.cpu().view(torch.int16).numpy().view(np.uint16)
    flat = x_bits.reshape(-1, 128)
    want, st = oracle.rope_fake_quant(flat, rows_per_token, positions, cos, sin, style, mode)
    return got.reshape(-1, 128), want, st, int(err.item())


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("name", ["tiny", "decode", "mtp", "prefill"])
def test_fake_quant_queries_and_keys(name, mode):
    w = wl.make(name)
    got, want, st, err = run_both(w.q, w.positions, w.cos, w.sin, w.rope_style, mode, w.H)
    assert st == 0 and err == 0
    assert_bytes_equal(got, want, f"{name} q fake quant mode {mode}")
    got, want, st, err = run_both(w.k, w.positions, w.cos, w.sin, w.rope_style, mode, 1)
    assert st == 0 and err == 0
    assert_bytes_equal(got, want, f"{name} k fake quant mode {mode}")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("style", [wl.ROPE_NEOX, wl.ROPE_INTERLEAVED])
def test_fake_quant_scales(style, mode):
    """Rows at scales 1e-3, 1, 40 and 1e4 (E4M3 saturation), zero rows and
    a ragged row count."""
    rng = np.random.Generator(np.random.PCG64(81 + style))
    cos, sin = wl.rope_tables(64)
    n = 333
    scales = rng.choice([1e-3, 1.0, 40.0, 1e4], size=n)
    x = rng.standard_normal((n, 128)) * scales[:, None]
    x[5] = 0.0
    bits = wl.to_bf16_bits(x)
    pos = rng.integers(0, 64, n).astype(np.int64)
    got, want, st, err = run_both(bits, pos, cos, sin, style, mode, 1)
    assert st == 0 and err == 0
    assert_bytes_equal(got, want, f"scales style {style} mode {mode}")


def test_fake_quant_bad_position_skips_row():
    cos, sin = wl.rope_tables(16)
    rng = np.random.Generator(np.random.PCG64(83))
    bits = wl.to_bf16_bits(rng.standard_normal((8, 128)))
    pos = np.array([0, 1, 99, 3, -1, 5, 6, 7], np.int64)
    x = bf16_dev(bits)
    out = torch.full((8, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    F().rope_fake_quant(x, dev(pos), dev(cos), dev(sin), scale_mode=1, out=out, err_flags=err)
    torch.cuda.synchronize()
    got = out.cpu().view(torch.int16).numpy().view(np.uint16)
    want = np.full((8, 128), wl.to_bf16_bits(np.float32(7.0)), np.uint16)
    st = oracle.rope_fake_quant(bits, 1, pos, cos, sin, 0, 1, out=want)[1]
    assert st == -1 and int(err.item()) == F().ERRFLAG_POSITION
    assert_bytes_equal(got, want, "bad positions")

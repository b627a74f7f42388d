"""GPU parity of the FP8 output mode (fp4idx_options.output_mode =
FP4IDX_OUTPUT_FP8) against the oracle on the same seeded inputs: the whole
8448-byte-page cache and the E4M3 query codes byte for byte, the weights
(each row's power-of-two scale folded in) within 1 ulp.  Source: "[HIP] Add
FP4 output mode to indexer_qk_rope_quant_and_cache" (aiter PR 5484),
Summary and API (the FP8 contract the FP4 mode extends)."""
import numpy as np
import pytest
import torch

import oracle
from fp4_sparse_attention_fp4idx_gb300 import workloads as wl
from tests.gpu_util import DeviceWorkload, F, assert_bytes_equal, assert_weights, dev

pytestmark = pytest.mark.gpu


def run_gpu(dw: DeviceWorkload, mode: str, ratio: int = 1, hadamard: bool = False):
    w = dw.w
    f = F()
    cache = dev(wl.fp8_sentinel_cache(w))
    if mode == "fused":
        qo, wt = f.indexer_prepass_fp8(dw.k, dw.gamma, dw.slots, cache, dw.q, dw.wt, dw.pos,
                                       dw.cos, dw.sin, eps=w.eps, rope_style=w.rope_style,
                                       compress_ratio=ratio, hadamard=hadamard,
                                       err_flags=dw.err)
    else:
        f.k_norm_rope_fp8_store(dw.k, dw.gamma, dw.pos, dw.cos, dw.sin, dw.slots, cache,
                                eps=w.eps, rope_style=w.rope_style, compress_ratio=ratio,
                                hadamard=hadamard, err_flags=dw.err)
        qo, wt = f.q_rope_fp8_weights(dw.q, dw.wt, dw.pos, dw.cos, dw.sin,
                                      rope_style=w.rope_style, hadamard=hadamard,
                                      err_flags=dw.err)
    torch.cuda.synchronize()
    return cache.cpu().numpy(), qo.cpu().numpy(), wt.cpu().numpy()


def run_ref(w: wl.Workload, ratio: int = 1, hadamard: bool = False):
    cache = wl.fp8_sentinel_cache(w)
    oracle.k_norm_rope_fp8_store(w.k, w.gamma, w.eps, w.positions, w.cos, w.sin, w.rope_style,
                                 w.slot_mapping, cache, compress_ratio=ratio, hadamard=hadamard)
    qo, wt, _ = oracle.q_rope_fp8_weights(w.q, w.w, w.positions, w.cos, w.sin, w.rope_style,
                                          hadamard=hadamard)
    return cache, qo, wt


def assert_fp8_same(name, got, want):
    assert_bytes_equal(got[0], want[0], f"{name} fp8 kv_cache")
    assert_bytes_equal(got[1], want[1], f"{name} fp8 q codes")
    assert_weights(got[2], want[2], f"{name} fp8 weights")


@pytest.mark.parametrize("mode", ["fused", "separate"])
@pytest.mark.parametrize("name", ["tiny", "tiny_gamma1", "decode", "mtp", "prefill"])
def test_fp8_parity(name, mode):
    w = wl.make(name)
    dw = DeviceWorkload(w)
    assert_fp8_same(name, run_gpu(dw, mode), run_ref(w))
    assert int(dw.err.item()) == 0


@pytest.mark.parametrize("ratio,hadamard", [(2, False), (4, True)])
@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_fp8_with_variants(name, ratio, hadamard):
    w = wl.make(name)
    dw = DeviceWorkload(w)
    assert_fp8_same(name, run_gpu(dw, "fused", ratio, hadamard), run_ref(w, ratio, hadamard))


def test_fp8_random_scales_both_styles():
    for style, seed in ((wl.ROPE_NEOX, 71), (wl.ROPE_INTERLEAVED, 72)):
        w = wl.make_random(257, 64, style, seed=seed)
        dw = DeviceWorkload(w)
        assert_fp8_same(w.name, run_gpu(dw, "fused"), run_ref(w))


def test_fp8_large_prefill_full_size():
    """The bench workload (T = 65536, H = 64) in the FP8 mode, one fused
    launch: the whole 16384-page cache, every query code and every weight
    against the oracle (run on all host cores)."""
    w = wl.make("large_prefill")
    dw = DeviceWorkload(w)
    got = run_gpu(dw, "fused")
    with oracle.threads():
        want = run_ref(w)
    assert_fp8_same("large_prefill", got, want)

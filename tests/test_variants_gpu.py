"""GPU parity of the pre-pass's stated variants (the fp4idx_options block of
include/fp4idx.h) against the oracle on the same seeded inputs: the paged
cache and the packed queries byte for byte, weights within 1 ulp.  Sources:
"DeepSeek-V4 FP4: fused_compress FP4 scatter + rmsnorm_rope_rotate FP4
KV-cache kernel" (aiter PR 4029), Changes (optional Hadamard rotation);
"dsv4.1: RoPE and FP4 packing kernels" (sglang PR 39656), Summary and
Verification (RoPE at the group's first position, compress ratios 1, 2, 4)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from fp4_sparse_attention_fp4idx_gb300 import workloads as wl
from tests.gpu_util import DeviceWorkload, F, assert_same, run_oracle

pytestmark = pytest.mark.gpu

VARIANTS = [(1, True), (2, False), (4, False), (4, True)]
IDS = [f"ratio{r}-{'hadamard' if h else 'plain'}" for r, h in VARIANTS]


@pytest.mark.parametrize("mode", ["fused", "separate"])
@pytest.mark.parametrize("ratio,hadamard", VARIANTS, ids=IDS)
@pytest.mark.parametrize("name", ["tiny", "tiny_gamma1", "decode", "mtp"])
def test_variant_parity(name, ratio, hadamard, mode):
    w = wl.make(name)
    dw = DeviceWorkload(w)
    gpu = dw.run(mode, compress_ratio=ratio, hadamard=hadamard)
    assert_same(w, gpu, run_oracle(w, compress_ratio=ratio, hadamard=hadamard))
    assert int(dw.err.item()) == 0


@pytest.mark.parametrize("style", [wl.ROPE_NEOX, wl.ROPE_INTERLEAVED])
def test_variant_random_both_styles(style):
    """Random rows at scales 1e-3 .. 1e3 with both RoPE styles, rotation and
    ratio 2 together, fused call."""
    w = wl.make_random(333, 32, style, seed=61)
    dw = DeviceWorkload(w)
    gpu = dw.run("fused", compress_ratio=2, hadamard=True)
    assert_same(w, gpu, run_oracle(w, compress_ratio=2, hadamard=True))


def test_prefill_hadamard_full():
    """The prefill workload (8,192 tokens, H = 64) with the rotation: the
    whole cache and every query output (the oracle on all host cores)."""
    w = wl.make("prefill")
    dw = DeviceWorkload(w)
    gpu = dw.run("fused", hadamard=True)
    with oracle.threads():
        ref = run_oracle(w, hadamard=True)
    assert_same(w, gpu, ref)


def test_default_options_match_plain_calls():
    """An explicit options block holding the defaults gives the bytes of the
    plain entry point."""
    w = wl.make("tiny")
    dw = DeviceWorkload(w)
    plain = dw.run("fused")
    f = F()
    opts = f.Options(1, 0)
    dw.reset_cache()
    T, H = w.T, w.H
    qf = torch.empty((T, H, 64), dtype=torch.uint8, device="cuda")
    qs = torch.empty((T, H, 4), dtype=torch.uint8, device="cuda")
    wt = torch.empty((T, H), dtype=torch.float32, device="cuda")
    p = ctypes.c_void_p
    st = f.lib().fp4idx_indexer_prepass_ex(
        p(dw.k.data_ptr()), dw.k.stride(0), p(dw.gamma.data_ptr()), w.eps, p(dw.slots.data_ptr()),
        p(dw.cache.data_ptr()), w.num_blocks, p(dw.q.data_ptr()), dw.q.stride(0), dw.q.stride(1),
        p(dw.wt.data_ptr()), dw.wt.stride(0), f.default_weight_scale(H), p(qf.data_ptr()),
        p(qs.data_ptr()), p(wt.data_ptr()), H, p(dw.pos.data_ptr()), p(dw.cos.data_ptr()),
        p(dw.sin.data_ptr()), w.max_pos, w.rope_style, T, ctypes.cast(ctypes.pointer(opts), p),
        None, p(torch.cuda.current_stream().cuda_stream))
    assert st == f.OK
    torch.cuda.synchronize()
    assert np.array_equal(dw.cache.cpu().numpy(), plain[0])
    assert np.array_equal(qf.cpu().numpy(), plain[1])

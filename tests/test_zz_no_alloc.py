"""GPU test of fp4idx_indexer_prepass_host_static, the host-buffer pre-pass
whose device staging is the library's static buffer: two calls in a row give
the oracle's bytes (weights within 1 ulp), the second call changes nothing in
the device's free memory (the buffer is a module global, and neither call
allocates), and a request larger than the buffer is refused with
ERR_SCRATCH.  The file is named to be collected last, and runs alone as
well."""
import numpy as np
import pytest
import torch

from fp4_sparse_attention_fp4idx_gb300 import workloads as wl
from tests.gpu_util import F, assert_bytes_equal, assert_weights, dev, run_oracle

pytestmark = pytest.mark.gpu


def host_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()


def host(a):
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


def _inputs(w):
    """The call's device-side inputs, made before any measurement."""
    gamma = torch.from_numpy(w.gamma.view(np.int16)).view(torch.bfloat16).cuda()
    return gamma, dev(w.cos), dev(w.sin)


def _call(w, d, cache, chunk, err=None):
    gamma, cos, sin = d
    return F().indexer_prepass_host_static(
        host_bf16(w.k), gamma, host(w.slot_mapping), cache, host_bf16(w.q), host_bf16(w.w),
        host(w.positions), cos, sin, eps=w.eps, rope_style=w.rope_style, chunk_tokens=chunk,
        err_flags=err)


def test_static_staging_twice_in_a_row():
    w = wl.make_random(700, 64, wl.ROPE_NEOX, seed=4242)
    rc, rqf, rqs, rwt = run_oracle(w)
    d = _inputs(w)
    free_between = None
    for call in range(2):
        cache = dev(w.cache_init)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        qf, qs, wt = _call(w, d, cache, chunk=256, err=err)  # 3 chunks, a ragged last one
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        assert_bytes_equal(cache.cpu().numpy(), rc, f"kv_cache (call {call})")
        assert_bytes_equal(qf.numpy(), rqf, f"q_fp4 (call {call})")
        assert_bytes_equal(qs.numpy(), rqs, f"q_scale (call {call})")
        assert_weights(wt.numpy(), rwt)
        assert int(err.item()) == 0
        if call == 1:
            free_between = free_before - free_after
    # the first call may load the library's module (and with it the static
    # buffer); the second allocates nothing
    assert free_between == 0, free_between


def test_static_staging_refuses_oversize_chunk():
    w = wl.make_random(2000, 64, wl.ROPE_NEOX, seed=4244)
    cache = dev(w.cache_init)
    with pytest.raises(F().Fp4idxError) as e:
        _call(w, _inputs(w), cache, chunk=2000)  # 2000 x 64 rows need ~85 MB of staging
    assert e.value.status == F().ERR_SCRATCH


def test_static_staging_default_chunk_fits_128_heads():
    """Without chunk_tokens the binding picks a chunk whose staging fits the
    static buffer (512 tokens at 128 heads), and the bytes are the oracle's."""
    w = wl.make_random(600, 128, wl.ROPE_INTERLEAVED, seed=4245)
    rc, rqf, rqs, rwt = run_oracle(w)
    d = _inputs(w)
    cache = dev(w.cache_init)
    gamma, cos, sin = d
    qf, qs, wt = F().indexer_prepass_host_static(
        host_bf16(w.k), gamma, host(w.slot_mapping), cache, host_bf16(w.q), host_bf16(w.w),
        host(w.positions), cos, sin, eps=w.eps, rope_style=w.rope_style)
    torch.cuda.synchronize()
    assert_bytes_equal(cache.cpu().numpy(), rc, "kv_cache")
    assert_bytes_equal(qf.numpy(), rqf, "q_fp4")
    assert_bytes_equal(qs.numpy(), rqs, "q_scale")
    assert_weights(wt.numpy(), rwt)

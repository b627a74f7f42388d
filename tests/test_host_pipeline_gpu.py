"""GPU parity of the host-buffer form of the fused pre-pass: inputs and
outputs in (pinned) host memory, tokens processed in chunks on three streams
with the uploads, launches and downloads overlapped.  The result must be the
oracle's, byte for byte (weights within 1 ulp), for chunk sizes that leave a
ragged last chunk, a single partial chunk, and chunks that reuse both staging
slots several times."""
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


@pytest.mark.parametrize("style", [wl.ROPE_NEOX, wl.ROPE_INTERLEAVED])
@pytest.mark.parametrize("T,H,chunk", [(300, 32, 64), (70, 64, 128), (257, 16, 17), (1, 32, 8)])
def test_host_pipeline_matches_oracle(T, H, chunk, style):
    w = wl.make_random(T, H, style, seed=500 + T + H + chunk)
    cache = dev(w.cache_init)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gamma = torch.from_numpy(w.gamma.view(np.int16)).view(torch.bfloat16).cuda()
    qf, qs, wt = F().indexer_prepass_host(
        host_bf16(w.k), gamma, host(w.slot_mapping), cache, host_bf16(w.q), host_bf16(w.w),
        host(w.positions), dev(w.cos), dev(w.sin), eps=w.eps, rope_style=w.rope_style,
        chunk_tokens=chunk, err_flags=err)
    torch.cuda.synchronize()
    assert not qf.is_cuda and qf.is_pinned()
    rc, rqf, rqs, rwt = run_oracle(w)
    assert_bytes_equal(cache.cpu().numpy(), rc, "kv_cache")
    assert_bytes_equal(qf.numpy(), rqf, "q_fp4")
    assert_bytes_equal(qs.numpy(), rqs, "q_scale")
    assert_weights(wt.numpy(), rwt)
    assert int(err.item()) == 0


def test_host_pipeline_repeated_calls_share_staging():
    """Two calls in a row with the same chunking reuse the staging buffers;
    the second call's results are as exact as the first's."""
    w = wl.make_random(200, 32, wl.ROPE_NEOX, seed=77)
    gamma = torch.from_numpy(w.gamma.view(np.int16)).view(torch.bfloat16).cuda()
    args = (host_bf16(w.k), gamma, host(w.slot_mapping))
    rc, rqf, rqs, rwt = run_oracle(w)
    for _ in range(2):
        cache = dev(w.cache_init)
        qf, qs, wt = F().indexer_prepass_host(
            *args, cache, host_bf16(w.q), host_bf16(w.w), host(w.positions), dev(w.cos),
            dev(w.sin), eps=w.eps, rope_style=w.rope_style, chunk_tokens=48)
        torch.cuda.synchronize()
        assert_bytes_equal(cache.cpu().numpy(), rc, "kv_cache")
        assert_bytes_equal(qf.numpy(), rqf, "q_fp4")
        assert_bytes_equal(qs.numpy(), rqs, "q_scale")
        assert_weights(wt.numpy(), rwt)


def test_host_pipeline_two_threads_share_staging():
    """Two host threads, each on its own stream, call the host-buffer pre-pass
    three times each with the same chunking (so they share the library's
    pipeline and the binding's staging buffer); every result is the
    oracle's.  The calls enqueue one at a time and each waits until the
    previous one no longer uses the staging."""
    import threading
    ws = [wl.make_random(180, 32, wl.ROPE_NEOX, seed=901),
          wl.make_random(150, 32, wl.ROPE_INTERLEAVED, seed=902)]
    refs = [run_oracle(w) for w in ws]
    errors = []

    def worker(w, ref):
        try:
            s = torch.cuda.Stream()
            gamma = torch.from_numpy(w.gamma.view(np.int16)).view(torch.bfloat16).cuda()
            cos, sin = dev(w.cos), dev(w.sin)
            args = (host_bf16(w.k), gamma, host(w.slot_mapping))
            for _ in range(3):
                with torch.cuda.stream(s):
                    cache = dev(w.cache_init)
                    s.synchronize()
                    qf, qs, wt = F().indexer_prepass_host(
                        *args, cache, host_bf16(w.q), host_bf16(w.w), host(w.positions), cos, sin,
                        eps=w.eps, rope_style=w.rope_style, chunk_tokens=40, stream=s)
                    s.synchronize()
                assert_bytes_equal(cache.cpu().numpy(), ref[0], "kv_cache")
                assert_bytes_equal(qf.numpy(), ref[1], "q_fp4")
                assert_bytes_equal(qs.numpy(), ref[2], "q_scale")
                assert_weights(wt.numpy(), ref[3])
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(w, r)) for w, r in zip(ws, refs)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors

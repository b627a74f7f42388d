"""GPU parity of the FP4 prefill MQA-logits scorer (through the C ABI)
against the fp64 oracle: -inf exactly where the oracle has -inf (outside
each token's key range), every finite logit within 2^-17 * sum_h |w| sum_d
|q k|.  Source: "[HIP] Add FP4 output mode to
indexer_qk_rope_quant_and_cache" (aiter PR 5484), Summary (the FP4 scorer
"and its prefill variant")."""
import numpy as np
import pytest
import torch

import oracle
from fp4_sparse_attention_fp4idx_gb300 import workloads as wl
from tests.gpu_util import (DeviceWorkload, DevicePrefillScorer, F, assert_logits_close,
                            dev, prefill_magnitude, prefill_oracle)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", sorted(wl.PREFILL_SCORER_CONFIGS))
def test_prefill_scorer_parity(name):
    pw = wl.make_prefill_scorer_config(name)
    ds = DevicePrefillScorer(pw)
    out = ds.run().cpu().numpy()
    want, st = prefill_oracle(pw)
    assert st == 0
    rel = assert_logits_close(out, want, prefill_magnitude(pw), name)
    assert int(ds.err.item()) == 0
    print(f"{name}: max |err| / (sum|w| sum|qk|) = {rel:.3g}")


def test_prefill_untouched_columns():
    """Columns >= num_keys of a wider logits buffer keep their bytes."""
    pw = wl.make_prefill_scorer_config("prefill_h64_edges")
    ds = DevicePrefillScorer(pw)
    buf = torch.full((pw.T, pw.num_keys + 29), 777.0, dtype=torch.float32, device="cuda")
    ds.run(logits=buf)
    host = buf.cpu().numpy()
    assert np.all(host[:, pw.num_keys:] == 777.0)
    want, _ = prefill_oracle(pw)
    assert_logits_close(host[:, :pw.num_keys], want, prefill_magnitude(pw), "wide")


def test_prefill_host_checks():
    f = F()
    pw = wl.make_prefill_scorer_config("prefill_tiny_causal")
    ds = DevicePrefillScorer(pw)
    lib = f.lib()
    out = torch.empty((pw.T, pw.num_keys), dtype=torch.float32, device="cuda")
    names = ["qf", "qs", "w", "cache", "nb", "nk", "ks", "ke", "out", "os", "T", "H", "err",
             "stream"]
    base = [ds.q_fp4.data_ptr(), ds.q_scale.data_ptr(), ds.weights.data_ptr(),
            ds.cache.data_ptr(), pw.num_blocks, pw.num_keys, ds.ks.data_ptr(), ds.ke.data_ptr(),
            out.data_ptr(), out.stride(0), pw.T, pw.H, None, None]

    def call(**over):
        a = list(base)
        for k, v in over.items():
            a[names.index(k)] = v
        return lib.fp4idx_mqa_logits_prefill(*a)

    assert call(H=48) == f.ERR_SHAPE
    assert call(H=288) == f.ERR_SHAPE
    assert call(H=160) == f.ERR_SHAPE
    assert call(nk=pw.num_blocks * 64 + 1) == f.ERR_SHAPE
    assert call(os=pw.num_keys - 1) == f.ERR_SHAPE
    assert call(qf=ds.q_fp4.data_ptr() + 8) == f.ERR_ALIGN
    assert call(ks=None) == f.ERR_NULL
    assert call(T=0) == f.OK and call(nk=0) == f.OK
    torch.cuda.synchronize()


def test_prefill_chunk_full_size_sampled():
    """The DeepSeek-shaped prefill chunk (4096 tokens x 64 heads against
    16384 keys, causal) in the bench's launch configuration: 24 tokens
    (both ends and random ones) against the oracle, the -inf triangle of every
    token everywhere."""
    pw = wl.make_prefill_scorer_chunk()
    ds = DevicePrefillScorer(pw)
    out = ds.run().cpu().numpy()
    assert int(ds.err.item()) == 0
    cols = np.arange(pw.num_keys)
    inside = (cols[None, :] >= pw.ks[:, None]) & (cols[None, :] < pw.ke[:, None])
    assert np.array_equal(np.isneginf(out), ~inside)
    rng = np.random.Generator(np.random.PCG64(5))
    toks = np.unique(np.concatenate([[0, 1, pw.T - 2, pw.T - 1], rng.choice(pw.T, 20, False)]))
    sub = wl.PrefillScorerWorkload("sub", len(toks), pw.H, pw.num_keys, pw.q_fp4[toks],
                                   pw.q_scale[toks], pw.weights[toks], pw.kv_cache, pw.ks[toks],
                                   pw.ke[toks])
    with oracle.threads():
        want, st = prefill_oracle(sub)
        mag = prefill_magnitude(sub)
    assert_logits_close(out[toks], want, mag, "prefill chunk sampled")


def test_prepass_then_prefill_scorer():
    """The CUDA pre-pass writes a 300-token chunk's keys to consecutive slots
    and packs its queries; the CUDA prefill scorer then scores them causally.
    Against the oracle pre-pass then the oracle prefill scorer, from the same
    seeded bf16 inputs (H = 64)."""
    w = wl.make_random(300, 64, wl.ROPE_NEOX, seed=57, max_pos=512)
    w.slot_mapping = np.arange(w.T, dtype=np.int64)
    w.num_blocks = -(-w.T // 64)
    w.cache_init = np.zeros((w.num_blocks, wl.PAGE_BYTES), np.uint8)
    dw = DeviceWorkload(w)
    cache_g, qf_g, qs_g, wt_g = dw.run("fused")
    cache_o = w.cache_init.copy()
    oracle.k_norm_rope_pack_store(w.k, w.gamma, w.eps, w.positions, w.cos, w.sin,
                                  w.rope_style, w.slot_mapping, cache_o)
    qf_o, qs_o, wt_o, _ = oracle.q_rope_pack_weights(w.q, w.w, w.positions, w.cos, w.sin,
                                                     w.rope_style)
    ks = np.zeros(w.T, np.int32)
    ke = np.arange(1, w.T + 1, dtype=np.int32)
    pw_o = wl.PrefillScorerWorkload("pipe", w.T, w.H, w.T, qf_o, qs_o, wt_o, cache_o, ks, ke)
    want, _ = prefill_oracle(pw_o)
    got = F().mqa_logits_prefill(dev(qf_g), dev(qs_g), dev(wt_g), dev(cache_g), dev(ks), dev(ke),
                                 w.T)
    torch.cuda.synchronize()
    assert_logits_close(got.cpu().numpy(), want, prefill_magnitude(pw_o), "prefill pipeline")

"""GPU parity of the FP4 paged MQA-logits scorer (through the C ABI) against
the fp64 oracle on the same seeded bytes: -inf exactly where the oracle has
-inf, every finite logit within 2^-17 * sum_h |w| sum_d |q k|.  Sources:
"[HIP] Add FP4 output mode to indexer_qk_rope_quant_and_cache" (aiter PR
5484), Verification (the FP4 scorer consuming the pre-pass's bytes, GLM-5.2
shapes, next_n 1 and 4)."""
import numpy as np
import pytest
import torch

import oracle
from fp4_sparse_attention_fp4idx_gb300 import workloads as wl
from tests.gpu_util import (DeviceScorer, DeviceWorkload, F, SCORER_TOL,
                            assert_logits_close, bf16_dev, dev, scorer_magnitude,
                            scorer_oracle)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", sorted(wl.SCORER_CONFIGS) + sorted(wl.SCORER_MANY))
def test_scorer_parity(name):
    sw = wl.make_scorer_config(name)
    got = DeviceScorer(sw)
    out = got.run().cpu().numpy()
    want, st = scorer_oracle(sw)
    assert st == 0
    rel = assert_logits_close(out, want, scorer_magnitude(sw), name)
    assert int(got.err.item()) == 0
    print(f"{name}: max |err| / (sum|w| sum|qk|) = {rel:.3g}")


def test_scorer_untouched_columns_and_rows():
    """Columns >= max_context of a wider logits buffer keep their bytes."""
    sw = wl.make_scorer_config("scorer_glm_next1")
    ds = DeviceScorer(sw)
    rows = sw.batch * sw.next_n
    buf = torch.full((rows, sw.max_context + 37), 12345.0, dtype=torch.float32, device="cuda")
    ds.run(logits=buf)
    host = buf.cpu().numpy()
    assert np.all(host[:, sw.max_context:] == 12345.0)
    want, _ = scorer_oracle(sw)
    assert_logits_close(host[:, :sw.max_context], want, scorer_magnitude(sw), "wide")


def test_scorer_bad_pages_flagged():
    """Block-table entries outside [0, num_blocks) below the context: those 64
    logits are -inf (as in the oracle), the PAGE flag is raised, nothing else
    changes."""
    sw = wl.make_scorer_config("scorer_glm_next1")
    sw.block_table[3, 2] = sw.num_blocks
    sw.block_table[4, 0] = -7
    ds = DeviceScorer(sw)
    out = ds.run().cpu().numpy()
    want, st = scorer_oracle(sw)
    assert st == -1
    assert np.all(np.isneginf(out[3, 128:192])) and np.all(np.isneginf(out[4, :64]))
    assert_logits_close(out, want, scorer_magnitude(sw), "bad pages")
    assert int(ds.err.item()) == F().ERRFLAG_PAGE


def test_scorer_context_edge_values():
    """Context lengths above max_context (clamped), negative (all -inf), zero,
    and exactly a tile boundary."""
    sw = wl.make_scorer("edges", 4, 2, 32, [384, 0, 128, 129], 300, seed=41)
    sw.context_lens[:] = [100000, -5, 128, 129]
    ds = DeviceScorer(sw)
    out = ds.run().cpu().numpy()
    want, st = scorer_oracle(sw)
    assert st == 0
    assert_logits_close(out, want, scorer_magnitude(sw), "edges")
    assert np.all(np.isneginf(out[2:4]))


def test_scorer_host_checks_on_device():
    f = F()
    sw = wl.make_scorer_config("scorer_tiny")
    ds = DeviceScorer(sw)
    lib = f.lib()
    out = torch.empty((sw.batch, sw.max_context), dtype=torch.float32, device="cuda")
    base = [ds.q_fp4.data_ptr(), ds.q_scale.data_ptr(), ds.weights.data_ptr(),
            ds.cache.data_ptr(), sw.num_blocks, ds.bt.data_ptr(), ds.bt.stride(0),
            ds.ctx.data_ptr(), out.data_ptr(), out.stride(0), sw.batch, 1, 32,
            sw.max_context, None, None]

    def call(**over):
        a = list(base)
        names = ["qf", "qs", "w", "cache", "nb", "bt", "bts", "ctx", "out", "os", "batch",
                 "next_n", "H", "max_ctx", "err", "stream"]
        for k, v in over.items():
            a[names.index(k)] = v
        return lib.fp4idx_paged_mqa_logits(*a)

    assert call(H=48) == f.ERR_SHAPE
    assert call(H=160) == f.ERR_SHAPE   # more heads than one segment holds
    assert call(H=288) == f.ERR_SHAPE
    assert call(next_n=0) == f.ERR_SHAPE
    assert call(os=sw.max_context - 1) == f.ERR_SHAPE
    assert call(bts=1) == f.ERR_SHAPE
    assert call(qf=ds.q_fp4.data_ptr() + 8) == f.ERR_ALIGN
    assert call(cache=ds.cache.data_ptr() + 4) == f.ERR_ALIGN
    assert call(bt=None) == f.ERR_NULL
    assert call(batch=0) == f.OK and call(max_ctx=0) == f.OK
    torch.cuda.synchronize()


def test_scorer_full_size_sampled():
    """The full decode workload (128 sequences, next_n 4, H 32, contexts up to
    65,536) in the bench's launch configuration; 12 sequences checked against
    the oracle on all host cores (the shortest, the longest and ten more),
    the -inf padding of all sequences checked everywhere."""
    sw = wl.make_scorer_decode()
    ds = DeviceScorer(sw)
    out = ds.run().cpu().numpy()
    assert int(ds.err.item()) == 0
    lens = sw.context_lens
    for b in range(sw.batch):
        r = slice(b * sw.next_n, (b + 1) * sw.next_n)
        assert np.all(np.isneginf(out[r, lens[b]:]))
        assert np.all(np.isfinite(out[r, :lens[b]]))
    rng = np.random.Generator(np.random.PCG64(78))
    seqs = sorted({int(np.argmin(lens)), int(np.argmax(lens)),
                   *rng.choice(sw.batch, 10, replace=False).tolist()})
    sub = sw.rows_of(seqs)
    with oracle.threads():
        want, st = scorer_oracle(sub)
        mag = scorer_magnitude(sub)
    assert st == 0
    assert_logits_close(out[sub.notes["rows"]], want, mag, "decode sampled")


def test_prepass_then_scorer_pipeline():
    """Pre-pass bytes feeding the scorer, each side on its own: the CUDA
    pre-pass then the CUDA scorer, against the oracle pre-pass then the oracle
    scorer, from the same seeded bf16 keys/queries (one sequence of 300
    tokens in shuffled pages, next_n 4 = its last 4 tokens, H = 32)."""
    w = wl.make_random(300, 32, wl.ROPE_NEOX, seed=51, max_pos=512)
    rng = np.random.Generator(np.random.PCG64(52))
    npages = -(-w.T // 64)
    perm = rng.permutation(npages + 2).astype(np.int64)
    slots = perm[np.arange(w.T) // 64] * 64 + np.arange(w.T) % 64
    w.slot_mapping = slots
    w.num_blocks = npages + 2
    w.cache_init = rng.integers(0, 256, size=(w.num_blocks, wl.PAGE_BYTES), dtype=np.uint8)
    dw = DeviceWorkload(w)
    cache_g, qf_g, qs_g, wt_g = dw.run("fused")
    cache_o = w.cache_init.copy()
    oracle.k_norm_rope_pack_store(w.k, w.gamma, w.eps, w.positions, w.cos, w.sin,
                                  w.rope_style, w.slot_mapping, cache_o)
    qf_o, qs_o, wt_o, _ = oracle.q_rope_pack_weights(w.q, w.w, w.positions, w.cos, w.sin,
                                                     w.rope_style)
    last = slice(w.T - 4, w.T)
    bt = perm[:npages].astype(np.int32)[None, :]
    ctx = np.array([w.T], np.int32)
    sw_o = wl.ScorerWorkload("pipe", 1, 4, 32, w.T, qf_o[last], qs_o[last], wt_o[last],
                             cache_o, bt, ctx)
    want, st = scorer_oracle(sw_o)
    assert st == 0
    got = F().paged_mqa_logits(dev(qf_g[last]), dev(qs_g[last]), dev(wt_g[last]),
                               dev(cache_g), dev(bt), dev(ctx), w.T, next_n=4)
    torch.cuda.synchronize()
    assert_logits_close(got.cpu().numpy(), want, scorer_magnitude(sw_o), "pipeline")

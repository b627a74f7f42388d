"""End-to-end accuracy of the FP4 indexer on the GPU: bf16 keys and queries
through the pre-pass (keys into a shuffled paged cache, queries packed with
their head weights) and then the paged scorer, all through the public API,
against the same pipeline in the oracle.  The intermediate bytes must match
exactly (the fp32 head weights within 1 ulp), the logits within the scorer's
error bound; on the logits the test
also asserts cosine >= 0.999999 and a top-64 overlap of 1.0 per row, and
prints how far the FP4 path is from the unquantised fp64 score (which sets
what the format itself costs, not a kernel error).  Sources: "[HIP] Add FP4
output mode to indexer_qk_rope_quant_and_cache" (aiter PR 5484), Verification
(GLM-5.2 shapes H 32, D 128, kv_block 64, next_n 1 and 4)."""
import numpy as np
import pytest

import bench
import oracle
from fp4_sparse_attention_fp4idx_gb300 import workloads as wl
from tests.gpu_util import F, SCORER_TOL, assert_weights

pytestmark = pytest.mark.gpu

CASES = [(32, 1), (32, 4), (64, 4)]


def oracle_pipeline(e):
    cache = np.zeros((e.num_blocks, wl.PAGE_BYTES), np.uint8)
    st = oracle.k_norm_rope_pack_store(e.k, e.gamma, e.eps, e.k_positions, e.cos, e.sin,
                                       e.rope_style, e.slot_mapping, cache)
    assert st == 0
    qf, qs, wt, st = oracle.q_rope_pack_weights(e.q, e.w, e.q_positions, e.cos, e.sin,
                                                e.rope_style)
    assert st == 0
    with oracle.threads():
        lo, st = oracle.paged_mqa_logits(qf, qs, wt, cache, e.block_table, e.context_lens,
                                         e.next_n, e.ctx)
        # sum_h |w| sum_d |q k| per logit: the scorer on sign-cleared operands
        mc = cache.copy()
        mc[:, :wl.KV_BLOCK * 64] &= 0x77
        mag, _ = oracle.paged_mqa_logits(qf & 0x77, qs, np.abs(wt), mc, e.block_table,
                                         e.context_lens, e.next_n, e.ctx)
    assert st == 0
    return lo, cache, qf, qs, wt, mag


@pytest.mark.parametrize("H,next_n", CASES)
def test_indexer_end_to_end(H, next_n):
    e = wl.make_indexer_e2e(next_n=next_n, H=H)
    got, g_cache, g_qf, g_qs, g_wt = bench.indexer_pipeline(F(), e, "cuda")
    want, o_cache, o_qf, o_qs, o_wt, mag = oracle_pipeline(e)

    assert np.array_equal(g_cache, o_cache), "paged cache bytes differ"
    assert np.array_equal(g_qf, o_qf) and np.array_equal(g_qs, o_qs), "query bytes differ"
    # fp32(w * H^-1/2 * 128^-1/2): the library rounds the scale to fp32 first,
    # the oracle forms the product in double (1 ulp apart at most)
    assert_weights(g_wt, o_wt)

    assert np.all(np.isfinite(got)) and np.all(np.isfinite(want))
    err = np.abs(got.astype(np.float64) - want)
    assert np.all(err <= SCORER_TOL * mag), float((err / np.maximum(mag, 1e-300)).max())

    vs_oracle = bench.score_agreement(got, want)
    assert vs_oracle["cosine"] >= 0.999999, vs_oracle
    assert vs_oracle["top64_overlap"] == 1.0, vs_oracle

    vs_truth = bench.score_agreement(got, bench.unquantised_logits(e))
    print(f"H={H} next_n={next_n}: vs oracle {vs_oracle}; vs unquantised fp64 {vs_truth}")
    # The format's own loss: FP4 keys and queries still rank like the exact
    # score (a sanity floor, far below what the seeded data gives).
    assert vs_truth["cosine"] > 0.95 and vs_truth["top64_overlap"] > 0.6, vs_truth

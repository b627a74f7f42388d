"""The bounded waits' timeout path on the GPU, without a fault: the testing
hook makes one launch leave out the copies of one work item of its first
CTA, so that CTA's waits run out after their 1 s limit.  That launch must
return normally with FP4IDX_ERRFLAG_TIMEOUT raised (and nothing else
raised), the context must stay usable, and the next, normal launch must give
the same bytes as a launch before it.  Covers the streaming pre-pass kernel
and the paged scorer."""
import numpy as np
import pytest
import torch

from fp4_sparse_attention_fp4idx_gb300 import workloads as wl
from tests.gpu_util import DeviceScorer, F, bf16_dev, dev

pytestmark = pytest.mark.gpu


def _prepass(w, cache, err):
    f = F()
    qf, qs, wt = f.indexer_prepass(bf16_dev(w.k), bf16_dev(w.gamma), dev(w.slot_mapping), cache,
                                   bf16_dev(w.q), bf16_dev(w.w), dev(w.positions), dev(w.cos),
                                   dev(w.sin), eps=w.eps, rope_style=w.rope_style,
                                   err_flags=err)
    torch.cuda.synchronize()
    return [x.cpu().numpy() for x in (cache, qf, qs, wt)]


def test_prepass_timeout_then_normal_launch():
    w = wl.make("prefill")  # H = 64 (the streaming kernel), ~55 units per CTA
    f = F()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = _prepass(w, dev(w.cache_init), err)
    assert int(err.item()) == 0
    cache = dev(w.cache_init)
    f.test_withhold_next(f.TEST_PREPASS, 1)  # CTA 0's second unit
    _prepass(w, cache, err)
    assert int(err.item()) == f.ERRFLAG_TIMEOUT
    err.zero_()
    got = _prepass(w, cache, err)  # the same cache: every slot rewritten
    assert int(err.item()) == 0
    for a, b in zip(got, ref):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_scorer_timeout_then_normal_launch():
    sw = wl.make_scorer_config("scorer_many_short")  # ~12 tiles per CTA
    ds = DeviceScorer(sw)
    ref = ds.run().cpu().numpy()
    assert int(ds.err.item()) == 0
    f = F()
    f.test_withhold_next(f.TEST_SCORER, 2)
    ds.run()
    assert int(ds.err.item()) == f.ERRFLAG_TIMEOUT
    ds.err.zero_()
    got = ds.run().cpu().numpy()
    assert int(ds.err.item()) == 0
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))

"""CPU checks of bench.py's multi-rank plumbing with two gloo ranks: the
barrier, the max over ranks, the weak-scaling value, and that only rank 0
runs and prints the reference (oracle) arm."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    ws, r, _ = bench.dist_env()
    d = bench.init_dist(ws, "gloo")
    bench.barrier(d)
    local_ms = 1.0 + rank  # rank 1 is the slow one
    m = bench.max_over_ranks(local_ms, d)
    results[rank] = (m, bench.weak_scaling_value(ws, 1000, m))
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(bench.argparse.Namespace(
            workload="tiny", ref_tokens=8, steps=1, warmup=0))
    results[rank + 10] = buf.getvalue()
    bench.barrier(d)
    dist.destroy_process_group()


def test_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_rank_main, args=(2, port, results), nprocs=2, join=True)
        res = dict(results)
    assert res[0][0] == res[1][0] == pytest.approx(2.0)
    assert res[0][1] == res[1][1] == pytest.approx(2 * 1000 / 2e-3)
    assert '"impl": "reference"' in res[10] and res[11] == ""


def test_weak_scaling_value_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.weak_scaling_value(1, 65536, 0.25) == pytest.approx(65536 / 0.25e-3)
    assert bench.max_over_ranks(3.5, None) == 3.5


def test_prepass_bytes_match_array_sizes():
    """The pre-pass roofline numerator recounted from the byte sizes of what
    one fused launch must read and write on a small workload: every query
    row, head weight, position and slot entry, gamma, the key rows that have
    a slot, the cos/sin rows of the distinct positions, and the oracle's
    outputs plus one 68-byte slot per stored key."""
    sys.path.insert(0, ROOT)
    import numpy as np

    import bench
    import oracle
    from fp4_sparse_attention_fp4idx_gb300 import workloads as wl
    w = wl.make_random(300, 32, wl.ROPE_NEOX, seed=5)
    qf, qs, wt, _ = oracle.q_rope_pack_weights(w.q, w.w, w.positions, w.cos, w.sin,
                                               w.rope_style)
    valid = w.slot_mapping >= 0
    pos = np.unique(w.positions)
    assert 0 < pos.size < w.T and 0 < valid.sum() < w.T  # both counts are exercised
    reads = (w.q.nbytes + w.w.nbytes + w.positions.nbytes + w.slot_mapping.nbytes
             + w.gamma.nbytes + w.k[valid].nbytes + w.cos[pos].nbytes + w.sin[pos].nbytes)
    slot_bytes = w.cache_init.shape[1] // wl.KV_BLOCK
    writes = qf.nbytes + qs.nbytes + wt.nbytes + int(valid.sum()) * slot_bytes
    assert bench.algorithmic_bytes(w, "fused")["fused"] == reads + writes


def test_scorer_bytes_match_array_sizes():
    """The scorer roofline numerator recounted from array sizes: the slots of
    the cached tokens below each context, the block-table entries of the
    pages they occupy, the packed queries, scales, weights and context
    lengths, and the fp32 logits including the -inf padding."""
    sys.path.insert(0, ROOT)
    import numpy as np

    import bench
    from fp4_sparse_attention_fp4idx_gb300 import workloads as wl
    sw = wl.make_scorer_config("scorer_glm_next4")
    slot_bytes = sw.kv_cache.shape[1] // wl.KV_BLOCK
    reads = sw.q_fp4.nbytes + sw.q_scale.nbytes + sw.weights.nbytes + sw.context_lens.nbytes
    for b in range(sw.batch):
        ctx = min(max(int(sw.context_lens[b]), 0), sw.max_context)
        pages = sw.block_table[b, :-(-ctx // wl.KV_BLOCK)] if ctx else sw.block_table[b, :0]
        reads += ctx * slot_bytes + pages.nbytes
    logits = np.empty((sw.batch * sw.next_n, sw.max_context), np.float32)
    assert bench.scorer_bytes(sw) == reads + logits.nbytes


def test_traffic_record_only_for_its_workload_and_mode():
    """A committed DRAM-counter record is reported only beside the workload
    and launch mode it was captured on, and only while its kernel's source
    is the one that was captured."""
    sys.path.insert(0, ROOT)
    import json

    import bench
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        d = json.load(f)
    for kernel, rec in d.items():
        name, mode = rec["workload_name"], rec.get("mode", "fused")
        assert bench.traffic_record(kernel, name + "_other", mode) is None
        assert bench.traffic_record(kernel, name, "separate") is None or mode == "separate"
        got = bench.traffic_record(kernel, name, mode)
        if got is not None:  # None only while the source differs from the capture's
            assert got["dram_bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
    assert bench.traffic_record("no_such_kernel", "large_prefill") is None

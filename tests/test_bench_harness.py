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

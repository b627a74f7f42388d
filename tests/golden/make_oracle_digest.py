"""Writes tiny_oracle_digest.txt: SHA-256 digests of the oracle's outputs on
the Tiny and Tiny-gamma-1 workloads.  Calls only the oracle (and the seeded
input generators); run it after a deliberate change of the oracle's
arithmetic, and name the passage that justifies the change in the commit.

    python tests/golden/make_oracle_digest.py
"""
import hashlib
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from fp4_sparse_attention_fp4idx_gb300 import workloads as wl  # noqa: E402

OUT = os.path.join(HERE, "tiny_oracle_digest.txt")


def compute() -> dict:
    out = {}
    for name in ("tiny", "tiny_gamma1"):
        w = wl.make(name)
        cache = w.cache_init.copy()
        oracle.k_norm_rope_pack_store(w.k, w.gamma, w.eps, w.positions, w.cos, w.sin,
                                      w.rope_style, w.slot_mapping, cache)
        qf, qs, wt, _ = oracle.q_rope_pack_weights(w.q, w.w, w.positions, w.cos, w.sin,
                                                   w.rope_style)
        for key, arr in (("cache", cache), ("q_fp4", qf), ("q_scale", qs), ("weights", wt)):
            out[f"{name}.{key}"] = hashlib.sha256(arr.tobytes()).hexdigest()
    return out


def read_committed() -> dict:
    d = {}
    with open(OUT) as f:
        for ln in f:
            ln = ln.split("#", 1)[0].strip()
            if ln:
                k, v = ln.split()
                d[k] = v
    return d


if __name__ == "__main__":
    with open(OUT, "w") as f:
        f.write("# SHA-256 of the oracle's outputs on the Tiny workloads; written by\n")
        f.write("# tests/golden/make_oracle_digest.py (calls only the oracle).\n")
        for k, v in compute().items():
            f.write(f"{k} {v}\n")
    print(open(OUT).read())

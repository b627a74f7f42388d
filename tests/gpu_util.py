"""Shared plumbing of the GPU parity tests: upload a workload, run the CUDA
path through the C ABI (via the binding), run the oracle on the same inputs,
and compare (bytes exactly, weights within 1 ulp)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from fp4_sparse_attention_fp4idx_gb300 import workloads as wl


def F():
    from fp4_sparse_attention_fp4idx_gb300 import fp4idx
    return fp4idx


def bf16_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


class DeviceWorkload:
    def __init__(self, w: wl.Workload, device="cuda"):
        self.w = w
        self.q = bf16_dev(w.q, device)
        self.wt = bf16_dev(w.w, device)
        self.k = bf16_dev(w.k, device)
        self.gamma = bf16_dev(w.gamma, device)
        self.pos = dev(w.positions, device)
        self.cos = dev(w.cos, device)
        self.sin = dev(w.sin, device)
        self.slots = dev(w.slot_mapping, device)
        self.cache = dev(w.cache_init, device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)

    def reset_cache(self):
        self.cache.copy_(torch.from_numpy(self.w.cache_init))

    def run(self, mode: str = "fused", compress_ratio: int = 1, hadamard: bool = False):
        """Returns (cache, q_fp4, q_scale, weights) as numpy arrays."""
        f = F()
        w = self.w
        self.reset_cache()
        if mode == "fused":
            qf, qs, wt = f.indexer_prepass(self.k, self.gamma, self.slots, self.cache, self.q,
                                           self.wt, self.pos, self.cos, self.sin, eps=w.eps,
                                           rope_style=w.rope_style, err_flags=self.err,
                                           compress_ratio=compress_ratio, hadamard=hadamard)
        else:
            f.k_norm_rope_pack_store(self.k, self.gamma, self.pos, self.cos, self.sin,
                                     self.slots, self.cache, eps=w.eps,
                                     rope_style=w.rope_style, err_flags=self.err,
                                     compress_ratio=compress_ratio, hadamard=hadamard)
            qf, qs, wt = f.q_rope_pack_weights(self.q, self.wt, self.pos, self.cos, self.sin,
                                               rope_style=w.rope_style, err_flags=self.err,
                                               hadamard=hadamard)
        torch.cuda.synchronize()
        return (self.cache.cpu().numpy(), qf.cpu().numpy(), qs.cpu().numpy(),
                wt.cpu().numpy())


def run_oracle(w: wl.Workload, tokens=None, compress_ratio: int = 1, hadamard: bool = False):
    """Oracle outputs; with `tokens`, the query side covers only those tokens
    (rows in the given order) while the key side always covers all tokens."""
    cache = w.cache_init.copy()
    oracle.k_norm_rope_pack_store(w.k, w.gamma, w.eps, w.positions, w.cos, w.sin,
                                  w.rope_style, w.slot_mapping, cache,
                                  compress_ratio=compress_ratio, hadamard=hadamard)
    if tokens is None:
        qf, qs, wt, _ = oracle.q_rope_pack_weights(w.q, w.w, w.positions, w.cos, w.sin,
                                                   w.rope_style, hadamard=hadamard)
    else:
        qf, qs, wt, _ = oracle.q_rope_pack_weights(w.q[tokens], w.w[tokens],
                                                   w.positions[tokens], w.cos, w.sin,
                                                   w.rope_style, hadamard=hadamard)
    return cache, qf, qs, wt


def assert_bytes_equal(got: np.ndarray, want: np.ndarray, what: str):
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        n = bad.shape[0]
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {n} bytes differ; first at {i}: "
                             f"got {got[i]:#04x} want {want[i]:#04x}")


def ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    ia = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    ib = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    ia = np.where(ia < 0, -(ia & 0x7FFFFFFF), ia)
    ib = np.where(ib < 0, -(ib & 0x7FFFFFFF), ib)
    return np.abs(ia - ib)


def assert_weights(got: np.ndarray, want: np.ndarray, what: str = "weights", max_ulp: int = 1):
    d = ulp_distance(got, want)
    assert d.max(initial=0) <= max_ulp, f"{what}: max ulp distance {d.max()}"


def assert_same(w: wl.Workload, gpu, ref, tokens=None):
    cache, qf, qs, wt = gpu
    rc, rqf, rqs, rwt = ref
    assert_bytes_equal(cache, rc, f"{w.name} kv_cache")
    if tokens is not None:
        qf, qs, wt = qf[tokens], qs[tokens], wt[tokens]
    assert_bytes_equal(qf, rqf, f"{w.name} q_fp4")
    assert_bytes_equal(qs, rqs, f"{w.name} q_scale")
    assert_weights(wt, rwt, f"{w.name} weights")


# ------------------------------------------------------------------ scorer
# A logit's fp32 error bound: 2^-17 * sum_h |w| * sum_d |q k| (the header's
# contract for fp4idx_paged_mqa_logits: fp32 rounding of <= 128 products in
# the tensor core and <= 128 weighted head terms, each <= 2^-24 relative).
SCORER_TOL = 2.0 ** -17


class DeviceScorer:
    def __init__(self, sw: wl.ScorerWorkload, device="cuda"):
        self.sw = sw
        self.q_fp4 = dev(sw.q_fp4, device)
        self.q_scale = dev(sw.q_scale, device)
        self.weights = dev(sw.weights, device)
        self.cache = dev(sw.kv_cache, device)
        self.bt = dev(sw.block_table, device)
        self.ctx = dev(sw.context_lens, device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)

    def run(self, logits=None):
        out = F().paged_mqa_logits(self.q_fp4, self.q_scale, self.weights, self.cache, self.bt,
                                   self.ctx, self.sw.max_context, next_n=self.sw.next_n,
                                   logits=logits, err_flags=self.err)
        torch.cuda.synchronize()
        return out


def scorer_oracle(sw: wl.ScorerWorkload):
    return oracle.paged_mqa_logits(sw.q_fp4, sw.q_scale, sw.weights, sw.kv_cache,
                                   sw.block_table, sw.context_lens, sw.next_n, sw.max_context)


def scorer_magnitude(sw: wl.ScorerWorkload) -> np.ndarray:
    """sum_h |w| * sum_d |q k| per logit: the oracle on sign-cleared inputs
    (every dot product is then >= 0, so ReLU passes it unchanged)."""
    cache = sw.kv_cache.copy()
    cache[:, :wl.KV_BLOCK * 64] &= 0x77
    out, _ = oracle.paged_mqa_logits(sw.q_fp4 & 0x77, sw.q_scale, np.abs(sw.weights), cache,
                                     sw.block_table, sw.context_lens, sw.next_n,
                                     sw.max_context)
    return out


def assert_logits_close(got: np.ndarray, want: np.ndarray, mag: np.ndarray, what: str):
    assert got.shape == want.shape, (what, got.shape, want.shape)
    ninf_w, ninf_g = np.isneginf(want), np.isneginf(got)
    assert np.array_equal(ninf_w, ninf_g), (what, "-inf pattern differs",
                                            np.argwhere(ninf_w != ninf_g)[:5])
    fin = ~ninf_w
    assert np.all(np.isfinite(got[fin])), (what, "non-finite logits")
    err = np.abs(got[fin].astype(np.float64) - want[fin].astype(np.float64))
    lim = SCORER_TOL * mag[fin].astype(np.float64)
    bad = err > lim
    assert not bad.any(), (what, int(bad.sum()), float(err[bad].max()),
                           np.argwhere(fin)[np.flatnonzero(bad)[:5]].tolist())
    return float((err / np.maximum(mag[fin], 1e-300)).max()) if err.size else 0.0


# ---------------------------------------------------------- prefill scorer
def prefill_oracle(pw: wl.PrefillScorerWorkload):
    return oracle.mqa_logits_prefill(pw.q_fp4, pw.q_scale, pw.weights, pw.kv_cache, pw.ks,
                                     pw.ke, pw.num_keys)


def prefill_magnitude(pw: wl.PrefillScorerWorkload) -> np.ndarray:
    """sum_h |w| * sum_d |q k| per logit (the oracle on sign-cleared inputs)."""
    cache = pw.kv_cache.copy()
    cache[:, :wl.KV_BLOCK * 64] &= 0x77
    out, _ = oracle.mqa_logits_prefill(pw.q_fp4 & 0x77, pw.q_scale, np.abs(pw.weights), cache,
                                       pw.ks, pw.ke, pw.num_keys)
    return out


class DevicePrefillScorer:
    def __init__(self, pw: wl.PrefillScorerWorkload, device="cuda"):
        self.pw = pw
        self.q_fp4 = dev(pw.q_fp4, device)
        self.q_scale = dev(pw.q_scale, device)
        self.weights = dev(pw.weights, device)
        self.cache = dev(pw.kv_cache, device)
        self.ks = dev(pw.ks, device)
        self.ke = dev(pw.ke, device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)

    def run(self, logits=None):
        out = F().mqa_logits_prefill(self.q_fp4, self.q_scale, self.weights, self.cache, self.ks,
                                     self.ke, self.pw.num_keys, logits=logits,
                                     err_flags=self.err)
        torch.cuda.synchronize()
        return out


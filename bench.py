"""Benchmark of the fused FP4 indexer pre-pass (keys + queries) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload large_prefill] [--mode fused|separate]

One step = the whole hot path over one batch: key RMSNorm/RoPE/FP4/paged
store for T tokens and query RoPE/FP4/pack/head weights for T x H rows, with
the inputs resident in HBM.  Prints ONE JSON line (rank 0).

Timing: W untimed warm-up steps (through the public Python API), then K
timed steps between a barrier and a device synchronisation.  Before every
timed step, outside its CUDA events: a buffer of twice the L2 size is
written (no step reads a previous step's data from L2), another such buffer
is read (so the flush's own dirty lines are written back before the step,
not inside it), and the GPU sleeps ~0.1 ms so the launch is queued before
the start event.  Timed launches call the C ABI with pre-converted
arguments.  Per-step device time comes from CUDA events on the launching
stream.  nvidia-smi samples SM clocks and throttle reasons during the timed
region.

The reference arm (--impl reference) times the CPU oracle on the host cores
on a bounded sample of the same workload; under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = ("tokens/s and achieved HBM GB/s (fraction of GB300 peak), "
          "fused indexer K+Q FP4 pack")
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------- bytes model
def algorithmic_bytes(w, mode: str) -> dict:
    """Bytes a step must move at minimum.  Per query row: 256 (q) + 2 (w) +
    64 (q_fp4) + 4 (q_scale) + 4 (weight); per token: 8 (position) + 8 (slot);
    per distinct position: 256 (cos+sin rows); per stored key row: 256 (k) +
    68 (slot); once: 256 (gamma).  The separate key call re-reads positions
    and cos/sin rows for its own rows."""
    T, H = w.T, w.H
    valid = (w.slot_mapping >= 0)
    n_valid = int(valid.sum())
    d_all = int(np.unique(w.positions).size)
    d_valid = int(np.unique(w.positions[valid]).size)
    q_call = T * H * (256 + 2 + 64 + 4 + 4) + T * 8 + 256 * d_all
    k_call = n_valid * (256 + 68 + 8) + T * 8 + 256 * d_valid + 256
    fused = T * H * (256 + 2 + 64 + 4 + 4) + T * 16 + 256 * d_all + n_valid * (256 + 68) + 256
    return {"q_call": q_call, "k_call": k_call, "fused": fused,
            "step": fused if mode == "fused" else q_call + k_call, "n_valid": n_valid}


def prepass_kernel_name(H: int) -> str:
    """The kernel a pre-pass launch runs, in every output mode and with or
    without the rotation: the streaming kernel when the head count is a
    multiple of 16, otherwise the per-warp kernel."""
    return "stream_kernel" if H % 16 == 0 else "prepass_kernel"


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def traffic_record(kernel: str, workload: str, mode: str = "fused"):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    counters were taken on another workload or launch mode, or the kernel's
    source file changed since."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        rec = d.get(kernel)
        if not rec or rec.get("workload_name") != workload or rec.get("mode", "fused") != mode:
            return None
        with open(os.path.join(ROOT, rec["source_file"]), "rb") as f:
            h = hashlib.sha256(f.read()).hexdigest()
        if rec.get("source_sha256") == h:
            return rec
    except Exception:
        pass
    return None


def spread(ms) -> dict:
    """Median, min, 90th percentile and mean of per-launch times (ms)."""
    a = np.asarray(list(ms), np.float64)
    return {"median": round(float(np.median(a)), 5), "min": round(float(a.min()), 5),
            "p90": round(float(np.percentile(a, 90)), 5), "mean": round(float(a.mean()), 5),
            "n": int(a.size)}


def time_launches(launch, flush, steps: int, warmup: int, stream) -> list:
    """CUDA-event time (ms) of `steps` launches on `stream`, the L2 flushed
    before each (outside its events), after `warmup` untimed launches."""
    import torch
    for _ in range(warmup):
        flush()
        launch()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        flush()
        a.record(stream)
        launch()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for ln in f:
                p = [x.strip() for x in ln.split(",")]
                if len(p) >= 9:
                    rows.append(p)
        os.unlink(self.path)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------ distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws: int, backend: str):
    import torch.distributed as dist
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if ws > 1 else None


def max_over_ranks(x: float, dist, device=None) -> float:
    """Max of a scalar over all ranks (identity when not distributed)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(world_size: int, tokens_per_rank: int, max_step_ms: float) -> float:
    """Whole-job tokens/s: every rank processes its own full batch (weak
    scaling, no data exchanged), and the slowest rank sets the step time."""
    return world_size * tokens_per_rank / (max_step_ms / 1e3)


def barrier(dist):
    if dist is not None:
        dist.barrier()


# --------------------------------------------------------------- our arm
def upload(w, device):
    import torch

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    def d(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    return dict(k=bf(w.k), gamma=bf(w.gamma), slots=d(w.slot_mapping), cache=d(w.cache_init),
                q=bf(w.q), w=bf(w.w), pos=d(w.positions), cos=d(w.cos), sin=d(w.sin))


def make_step(F, D, w, mode, outs):
    """A step through the public API (argument checks included)."""
    qf, qs, wt = outs

    def step():
        if mode == "fused":
            F.indexer_prepass(D["k"], D["gamma"], D["slots"], D["cache"], D["q"], D["w"],
                              D["pos"], D["cos"], D["sin"], eps=w.eps, rope_style=w.rope_style,
                              q_fp4=qf, q_scale=qs, weights=wt)
        else:
            F.k_norm_rope_pack_store(D["k"], D["gamma"], D["pos"], D["cos"], D["sin"],
                                     D["slots"], D["cache"], eps=w.eps, rope_style=w.rope_style)
            F.q_rope_pack_weights(D["q"], D["w"], D["pos"], D["cos"], D["sin"],
                                  rope_style=w.rope_style, q_fp4=qf, q_scale=qs, weights=wt)
    return step


def make_raw_launches(F, D, w, mode, outs):
    """The same C-ABI calls with every argument converted once, so that the
    host-side cost between a start event and the launch is one foreign
    call.  Returns a list of callables (one per launch of a step)."""
    import torch
    L = F.lib()
    qf, qs, wt = outs
    T, H = w.T, w.H
    ws = F.default_weight_scale(H)
    st = torch.cuda.current_stream().cuda_stream
    p = {k: v.data_ptr() for k, v in D.items()}
    if mode == "fused":
        args = (p["k"], 128, p["gamma"], w.eps, p["slots"], p["cache"], w.num_blocks, p["q"],
                H * 128, 128, p["w"], H, ws, qf.data_ptr(), qs.data_ptr(), wt.data_ptr(), H,
                p["pos"], p["cos"], p["sin"], w.max_pos, w.rope_style, T, None, st)
        fn = L.fp4idx_indexer_prepass
        return [lambda: _ok(F, fn(*args))]
    kargs = (p["k"], 128, p["gamma"], w.eps, p["pos"], p["cos"], p["sin"], w.max_pos,
             w.rope_style, p["slots"], p["cache"], w.num_blocks, T, None, st)
    qargs = (p["q"], H * 128, 128, p["w"], H, ws, p["pos"], p["cos"], p["sin"], w.max_pos,
             w.rope_style, qf.data_ptr(), qs.data_ptr(), wt.data_ptr(), T, H, None, st)
    kf, qfn = L.fp4idx_k_norm_rope_pack_store, L.fp4idx_q_rope_pack_weights
    return [lambda: _ok(F, kf(*kargs)), lambda: _ok(F, qfn(*qargs))]


def _ok(F, status):
    if status != 0:
        raise RuntimeError(F.status_string(status))


class L2Flush:
    """Writes a buffer of twice the L2 size (evicting every input line), then
    reads a second such buffer so that the flush's own dirty lines are
    written back before the timed launch rather than inside it; then keeps
    the GPU busy for a while so that the next launch is queued before its
    start event (no host-side gap inside the timed interval)."""

    def __init__(self, device):
        import torch
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        n = max(2 * l2, 256 << 20) // 4
        self.w = torch.empty(n, dtype=torch.float32, device=device)
        self.r = torch.zeros(n, dtype=torch.float32, device=device)
        self.bytes = 2 * l2

    def __call__(self):
        import torch
        self.w.zero_()
        self.r.sum()
        torch.cuda._sleep(200_000)  # ~0.1 ms of GPU time at 2 GHz


def time_device(F, w, D, mode, steps, warmup, flush, dist=None, sampler=None):
    """Per-step CUDA-event times (ms) of the whole step and, in separate mode,
    of each launch; an L2 flush precedes every step, outside the events."""
    import torch
    dev = D["q"].device
    T, H = w.T, w.H
    outs = (torch.empty((T, H, 64), dtype=torch.uint8, device=dev),
            torch.empty((T, H, 4), dtype=torch.uint8, device=dev),
            torch.empty((T, H), dtype=torch.float32, device=dev))
    step = make_step(F, D, w, mode, outs)
    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()
    launches = make_raw_launches(F, D, w, mode, outs)
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(dist)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.1)
    t0 = time.perf_counter()
    for i in range(steps):
        flush()
        a, m, b = ev[i]
        a.record(stream)
        launches[0]()
        if len(launches) > 1:
            m.record(stream)
            launches[1]()
        b.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier(dist)
    clocks = sampler.stop() if sampler else None
    step_ms = [a.elapsed_time(b) for a, _, b in ev]
    res = {"step_ms": step_ms, "wall_s": wall, "clocks": clocks}
    if mode != "fused":
        res["k_ms"] = [a.elapsed_time(m) for a, m, _ in ev]
        res["q_ms"] = [m.elapsed_time(b) for _, m, b in ev]
    return res


def time_e2e(F, w, D, mode, steps):
    """Through the public API with host buffers: per step, the step's inputs
    (q, w, k, positions, slot mapping) come from pinned host memory and the
    query outputs go back to pinned host memory.  Fused mode uses
    indexer_prepass_host (chunked, uploads / launches / downloads
    overlapped); separate mode copies, runs the two calls and copies back.
    The cos/sin tables, gamma and the paged cache stay resident on the
    device."""
    import torch
    dev = D["q"].device
    names = ("q", "w", "k", "pos", "slots")
    host = {n: D[n].cpu().pin_memory() for n in names}
    T, H = w.T, w.H
    outs = (torch.empty((T, H, 64), dtype=torch.uint8, device=dev),
            torch.empty((T, H, 4), dtype=torch.uint8, device=dev),
            torch.empty((T, H), dtype=torch.float32, device=dev))
    hout = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    step = make_step(F, D, w, mode, outs)
    stream = torch.cuda.current_stream()
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = sum(o.numel() * o.element_size() for o in outs)

    def one():
        if mode == "fused":
            F.indexer_prepass_host(host["k"], D["gamma"], host["slots"], D["cache"], host["q"],
                                   host["w"], host["pos"], D["cos"], D["sin"], eps=w.eps,
                                   rope_style=w.rope_style, q_fp4=hout[0], q_scale=hout[1],
                                   weights=hout[2])
            return
        for n in names:
            D[n].copy_(host[n], non_blocking=True)
        step()
        for o, h in zip(outs, hout):
            h.copy_(o, non_blocking=True)

    one()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        one()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps, h2d, d2h


# ------------------------------------------------------------- variants
def run_variants(F, w, D, dev, peak, flush, steps: int = 100, warmup: int = 5) -> dict:
    """The fused pre-pass with the stated variants (the fp4idx_options block)
    on the same workload: CUDA-event time per launch, L2 flushed before each,
    and the fraction of the measured HBM peak (the algorithmic bytes do not
    change with the options)."""
    import ctypes
    import torch
    T, H = w.T, w.H
    qf = torch.empty((T, H, 64), dtype=torch.uint8, device=dev)
    qs = torch.empty((T, H, 4), dtype=torch.uint8, device=dev)
    wt = torch.empty((T, H), dtype=torch.float32, device=dev)
    p = {k: v.data_ptr() for k, v in D.items()}
    st = torch.cuda.current_stream()
    fn = F.lib().fp4idx_indexer_prepass_ex
    nbytes4 = algorithmic_bytes(w, "fused")["fused"]
    # FP8 mode: per query row 256 + 2 + 128 (codes) + 4 (weight), per stored
    # key row 256 + 132 (slot); no exponent words for queries
    nv = algorithmic_bytes(w, "fused")["n_valid"]
    nbytes8 = nbytes4 + T * H * (128 - 64 - 4) + nv * (132 - 68)
    q8 = torch.empty((T, H, 128), dtype=torch.uint8, device=dev)
    cache8 = torch.zeros((w.num_blocks, F.FP8_PAGE_BYTES), dtype=torch.uint8, device=dev)
    out = {}
    for name, ratio, had, mode in (("hadamard", 1, 1, 0), ("compress_ratio_4", 4, 0, 0),
                                   ("compress_ratio_4_hadamard", 4, 1, 0), ("fp8", 1, 0, 1),
                                   ("fp8_hadamard", 1, 1, 1)):
        opts = ctypes.cast(ctypes.pointer(F.Options(ratio, had, mode)), ctypes.c_void_p)
        nbytes = nbytes8 if mode else nbytes4
        args = (p["k"], 128, p["gamma"], w.eps, p["slots"],
                cache8.data_ptr() if mode else p["cache"], w.num_blocks, p["q"],
                H * 128, 128, p["w"], H, F.default_weight_scale(H),
                q8.data_ptr() if mode else qf.data_ptr(), None if mode else qs.data_ptr(),
                wt.data_ptr(), H, p["pos"], p["cos"], p["sin"], w.max_pos,
                w.rope_style, T, opts, None, st.cuda_stream)
        sp = spread(time_launches(lambda: _ok(F, fn(*args)), flush, steps, warmup, st))
        ms = sp["median"]
        gbs = nbytes / (ms / 1e3) / 1e9
        out[name] = {"ms_per_launch": ms, "ms_spread": sp,
                     "tokens_per_s": round(T / (ms / 1e3), 1),
                     "gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
                     "algorithmic_bytes_per_launch": nbytes,
                     "kernel": prepass_kernel_name(H)}
    # The torch-shaped RoPE + FP4 fake quantisation of the workload's queries
    # (T*H rows): 256 B read + 256 B written per row, 8 B of position per
    # token, 256 B of cos/sin per distinct position.
    qo = torch.empty((T, H, 128), dtype=torch.bfloat16, device=dev)
    fq = F.lib().fp4idx_rope_fake_quant
    nbytes = T * H * 512 + T * 8 + 256 * int(np.unique(w.positions).size)
    for name, mode in (("fake_quant_ue8m0_32", 0), ("fake_quant_e4m3_16", 1)):
        args = (p["q"], 128, H, p["pos"], p["cos"], p["sin"], w.max_pos, w.rope_style, mode,
                qo.data_ptr(), T * H, None, st.cuda_stream)
        sp = spread(time_launches(lambda: _ok(F, fq(*args)), flush, steps, warmup, st))
        ms = sp["median"]
        gbs = nbytes / (ms / 1e3) / 1e9
        out[name] = {"ms_per_launch": ms, "ms_spread": sp,
                     "rows_per_s": round(T * H / (ms / 1e3), 1),
                     "gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
                     "algorithmic_bytes_per_launch": nbytes, "kernel": "fake_quant_kernel"}
    return out


# ------------------------------------------------------------------ scorer
def scorer_bytes(sw) -> int:
    """Bytes one scorer launch must move at minimum: per cached token below
    its context, its 68-byte slot; per used page, its 4-byte block-table
    entry; per query row, 64 + 4 bytes of packed query and a 4-byte weight;
    per sequence its context length; and the fp32 logits written, -inf
    padding included (batch * next_n * max_context * 4)."""
    ctx = np.minimum(np.maximum(sw.context_lens.astype(np.int64), 0), sw.max_context)
    pages = -(-ctx // 64)
    rows = sw.batch * sw.next_n
    return int(ctx.sum() * 68 + pages.sum() * 4 + rows * sw.H * 72 + sw.batch * 4
               + rows * sw.max_context * 4)


def prefill_scorer_bytes(pw) -> int:
    """Bytes one prefill-scorer launch must move at minimum: every key's
    68-byte slot once, per query row 64 + 4 + 4 bytes, per token its two
    int32 range bounds, and the fp32 logits written (num_tokens * num_keys
    * 4, -inf outside the ranges included)."""
    return int(pw.num_keys * 68 + pw.T * pw.H * 72 + pw.T * 8 + pw.T * pw.num_keys * 4)


# SM clock for the ALU peak: the part's maximum (the bench's clock samples
# show it is held under load, and the record reports them).
SM_MAX_MHZ = 2070.0


def alu_peak_gops(dev) -> float:
    """fp32 lane operations per second the SMs can issue: SMs x 128 lanes x
    the maximum SM clock (one warp instruction per cycle per sub-partition),
    in Gop/s."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    return sms * 128 * SM_MAX_MHZ * 1e6 / 1e9


def _scorer_record(name, ms_list, nbytes, flops, peak, extra, alu=None):
    """alu: (lane ops per launch, peak Gop/s) for a launch bound by its
    epilogue arithmetic rather than by HBM; the HBM figures are kept beside."""
    sp = spread(ms_list)
    ms = sp["median"]
    achieved = nbytes / (ms / 1e3) / 1e9
    tr = traffic_record(name, extra.get("workload"))
    rec = dict(extra)
    hbm = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
           "unit": "GB/s", "frac": round(achieved / peak, 4), "kernel": name,
           "algorithmic_bytes_per_launch": nbytes,
           "traffic": tr["dram_bytes_per_launch"] if tr else None}
    if alu is None:
        roof = hbm
    else:
        ops, alu_peak = alu
        got = ops / (ms / 1e3) / 1e9
        roof = {"bound": "alu", "achieved": round(got, 1), "peak": round(alu_peak, 1),
                "unit": "Gop/s", "frac": round(got / alu_peak, 4), "kernel": name,
                "algorithmic_ops_per_launch": int(ops),
                "ops": "per (key, query row): max(0, x) and half of an f32x2 fma",
                "peak_kind": "derived: SMs x 128 fp32 lanes x 2070 MHz",
                "hbm": {k: hbm[k] for k in ("achieved", "peak", "unit", "frac",
                                            "algorithmic_bytes_per_launch", "traffic")}}
    rec.update({
        "ms_per_launch": ms, "ms_spread": sp, "roofline": roof,
        "mxf4_tflops": round(flops / (ms / 1e3) / 1e12, 1),
        "l2": "flushed before every launch, outside the CUDA events"})
    return rec


def run_decode_scorer(F, sw, dev, peak, flush, steps: int, warmup: int = 5) -> dict:
    """One paged-scorer workload: CUDA-event time per launch and its HBM
    roofline (algorithmic bytes count every cached key once, also where a
    sequence's query rows are scored in several groups)."""
    import torch

    def d(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    qf, qs, wt, cache = d(sw.q_fp4), d(sw.q_scale), d(sw.weights), d(sw.kv_cache)
    bt, ctx = d(sw.block_table), d(sw.context_lens)
    rows = sw.batch * sw.next_n
    out = torch.empty((rows, sw.max_context), dtype=torch.float32, device=dev)
    F.paged_mqa_logits(qf, qs, wt, cache, bt, ctx, sw.max_context, next_n=sw.next_n, logits=out)
    torch.cuda.synchronize()
    fn = F.lib().fp4idx_paged_mqa_logits
    stream = torch.cuda.current_stream()
    args = (qf.data_ptr(), qs.data_ptr(), wt.data_ptr(), cache.data_ptr(), sw.num_blocks,
            bt.data_ptr(), bt.stride(0), ctx.data_ptr(), out.data_ptr(), out.stride(0),
            sw.batch, sw.next_n, sw.H, sw.max_context, None, stream.cuda_stream)
    ms = time_launches(lambda: _ok(F, fn(*args)), flush, steps, warmup, stream)
    ctx_tokens = int(np.minimum(np.maximum(sw.context_lens, 0), sw.max_context).sum())
    med = float(np.median(ms))
    groups = max(1, -(-sw.next_n * sw.H // 128))
    return _scorer_record("scorer_kernel", ms, scorer_bytes(sw),
                          2.0 * 128 * sw.next_n * sw.H * ctx_tokens, peak, {
        "workload": sw.name, "batch": sw.batch, "next_n": sw.next_n, "H": sw.H,
        "max_context": sw.max_context, "cached_tokens": ctx_tokens,
        "kv_cache_bytes": int(sw.kv_cache.nbytes), "launches": steps,
        "query_groups_per_sequence": groups,
        "scored_keys_per_s": round(ctx_tokens * sw.next_n / (med / 1e3), 1)})


def run_prefill_scorer(F, pw, dev, peak, flush, steps: int, warmup: int = 5) -> dict:
    """The prefill scorer on a prefill chunk: CUDA-event time per launch and
    its HBM roofline (algorithmic bytes count every key once)."""
    import torch

    def d(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    qf, qs, wt, cache = d(pw.q_fp4), d(pw.q_scale), d(pw.weights), d(pw.kv_cache)
    ks, ke = d(pw.ks), d(pw.ke)
    out = torch.empty((pw.T, pw.num_keys), dtype=torch.float32, device=dev)
    F.mqa_logits_prefill(qf, qs, wt, cache, ks, ke, pw.num_keys, logits=out)
    torch.cuda.synchronize()
    fn = F.lib().fp4idx_mqa_logits_prefill
    stream = torch.cuda.current_stream()
    args = (qf.data_ptr(), qs.data_ptr(), wt.data_ptr(), cache.data_ptr(), pw.num_blocks,
            pw.num_keys, ks.data_ptr(), ke.data_ptr(), out.data_ptr(), out.stride(0), pw.T,
            pw.H, None, stream.cuda_stream)
    ms = time_launches(lambda: _ok(F, fn(*args)), flush, steps, warmup, stream)
    lo = np.clip(pw.ks.astype(np.int64), 0, pw.num_keys)
    hi = np.clip(pw.ke.astype(np.int64), 0, pw.num_keys)
    scored = int(np.maximum(hi - lo, 0).sum())
    med = float(np.median(ms))
    # The head sums' ALU work: per (key, query row) a max and half an f32x2
    # fma, i.e. 1.5 lane operations.
    alu = (1.5 * pw.H * scored, alu_peak_gops(dev))
    return _scorer_record("scorer_kernel", ms, prefill_scorer_bytes(pw),
                          2.0 * 128 * pw.H * scored, peak, alu=alu, extra={
        "workload": pw.name, "T": pw.T, "H": pw.H, "num_keys": pw.num_keys,
        "scored_pairs": scored, "launches": steps,
        "scored_keys_per_s": round(scored / (med / 1e3), 1)})


def run_scorer(F, dev, peak, flush, steps: int) -> dict:
    """The FP4 scorer on three workloads: GLM-5.2-style decode (H 32,
    next_n 4, 128 sequences up to 64K tokens), DeepSeek-style decode with
    H 64 and next_n 4 (256 query rows per sequence, scored in two groups of
    128), and a DeepSeek-shaped prefill chunk (4096 query tokens, 16384
    keys, causal)."""
    from fp4_sparse_attention_fp4idx_gb300 import workloads as wl
    out = {"decode": run_decode_scorer(F, wl.make_scorer_decode(), dev, peak, flush, steps)}
    out["decode_h64_next4"] = run_decode_scorer(
        F, wl.make_scorer_decode(batch=64, H=64, name="scorer_decode_h64"), dev, peak, flush,
        steps)
    out["prefill_chunk"] = run_prefill_scorer(F, wl.make_prefill_scorer_chunk(), dev, peak,
                                              flush, max(20, steps // 4))
    return out


# ------------------------------------------------------------ accuracy
def unquantised_logits(e) -> np.ndarray:
    """The indexer score without any quantisation, in fp64: keys RMSNorm'd
    (gamma, eps) and rotated, queries rotated (exact angles p * 10000^(-2i/64)
    on dims 0..63), then sum_h w * max(0, q_h . k) with the head weights
    w * H^-1/2 * 128^-1/2.  Logits [batch*next_n, ctx]."""
    f = lambda b: (np.asarray(b, np.uint32) << 16).view(np.float32).astype(np.float64)
    i = np.arange(32, dtype=np.float64)
    inv = 10000.0 ** (-2.0 * i / 64)

    def rope(x, pos):
        th = pos[:, None].astype(np.float64) * inv[None, :]
        c, s_ = np.cos(th), np.sin(th)
        if x.ndim == 3:
            c, s_ = c[:, None, :], s_[:, None, :]
        y = x.copy()
        if e.rope_style == 0:
            a, b = x[..., :32], x[..., 32:64]
            y[..., :32], y[..., 32:64] = a * c - b * s_, b * c + a * s_
        else:
            a, b = x[..., 0:64:2], x[..., 1:64:2]
            y[..., 0:64:2], y[..., 1:64:2] = a * c - b * s_, b * c + a * s_
        return y

    k = f(e.k)
    k = k / np.sqrt((k * k).mean(axis=1, keepdims=True) + e.eps) * f(e.gamma)[None, :]
    k = rope(k, e.k_positions)
    q = rope(f(e.q), e.q_positions)
    w = f(e.w) / np.sqrt(e.H * 128.0)
    out = np.empty((e.batch * e.next_n, e.ctx))
    for b in range(e.batch):
        kb = k[b * e.ctx:(b + 1) * e.ctx]
        for j in range(e.next_n):
            t = b * e.next_n + j
            dots = q[t] @ kb.T  # [H, ctx]
            out[t] = (w[t][:, None] * np.maximum(dots, 0.0)).sum(axis=0)
    return out


def score_agreement(got: np.ndarray, ref: np.ndarray, k: int = 64) -> dict:
    """Cosine similarity of two logit arrays (over all entries), the mean
    top-k overlap per row (a pick counts when its reference value reaches the
    reference's k-th largest, so ties do not count against it), and the max
    absolute difference."""
    g, r = got.astype(np.float64).ravel(), ref.astype(np.float64).ravel()
    cos = float(g @ r / (np.linalg.norm(g) * np.linalg.norm(r)))
    ov = []
    for gr, rr in zip(got, ref):
        kk = min(k, rr.size)
        thresh = np.partition(rr, -kk)[-kk]
        picks = np.argpartition(gr, -kk)[-kk:]
        ov.append(float(np.mean(rr[picks] >= thresh)))
    return {"cosine": round(cos, 7), f"top{k}_overlap": round(float(np.mean(ov)), 4),
            "max_abs_err": float(np.max(np.abs(g - r)))}


def indexer_pipeline(F, e, device):
    """The whole path on the GPU through the public API: keys into the paged
    cache, queries packed with their head weights, then the paged scorer.
    Returns (logits [batch*next_n, ctx] fp32, cache, q_fp4, q_scale, weights)
    as numpy arrays."""
    import torch

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    def d(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    cache = torch.zeros((e.num_blocks, F.PAGE_BYTES), dtype=torch.uint8, device=device)
    cs, sn = d(e.cos), d(e.sin)
    F.k_norm_rope_pack_store(bf(e.k), bf(e.gamma), d(e.k_positions), cs, sn, d(e.slot_mapping),
                             cache, eps=e.eps, rope_style=e.rope_style)
    qf, qs, wt = F.q_rope_pack_weights(bf(e.q), bf(e.w), d(e.q_positions), cs, sn,
                                       rope_style=e.rope_style)
    logits = F.paged_mqa_logits(qf, qs, wt, cache, d(e.block_table), d(e.context_lens), e.ctx,
                                next_n=e.next_n)
    torch.cuda.synchronize()
    return tuple(x.cpu().numpy() for x in (logits, cache, qf, qs, wt))


def run_accuracy(F, device) -> dict:
    """The FP4 indexer path (pre-pass then scorer, all on the GPU) against
    the unquantised fp64 score, at GLM-5.2 shapes (H 32, D 128, kv_block 64),
    next_n 1 and 4: 4 sequences of 2048 tokens."""
    from fp4_sparse_attention_fp4idx_gb300 import workloads as wl
    out = {}
    for nn in (1, 4):
        e = wl.make_indexer_e2e(next_n=nn)
        got = indexer_pipeline(F, e, device)[0]
        out[f"next_n_{nn}"] = score_agreement(got, unquantised_logits(e))
    out["reference"] = ("unquantised fp64 indexer score from the same bf16 inputs (RMSNorm, "
                        "RoPE at exact angles, no FP4 rounding); the FP4 path against its own "
                        "oracle is held to cosine >= 0.999999 and top-64 overlap 1.0 by "
                        "tests/test_e2e_accuracy_gpu.py")
    return out


def _oracle_rate(w, S: int) -> float:
    """Seconds the oracle takes for the keys and queries of the first S
    tokens of the workload."""
    import oracle
    cache = w.cache_init.copy()
    t0 = time.perf_counter()
    oracle.k_norm_rope_pack_store(w.k[:S], w.gamma, w.eps, w.positions[:S], w.cos, w.sin,
                                  w.rope_style, w.slot_mapping[:S], cache)
    oracle.q_rope_pack_weights(w.q[:S], w.w[:S], w.positions[:S], w.cos, w.sin, w.rope_style)
    return time.perf_counter() - t0


def _oracle_sample(w, budget_s: float):
    """(S, seconds): S grown by 4x from 64 tokens until a run takes about a
    quarter of budget_s."""
    S = 64
    while True:
        dt = _oracle_rate(w, S)
        if dt * 4 > budget_s or S >= w.T:
            return S, dt
        S = min(w.T, S * 4)


def cpu_baseline(w, budget_s: float = 12.0):
    """The oracle as it stands on the host cores: on all of them (its token
    loops run in parallel; this is the reported value) and on one, each on
    the first S tokens of the workload (keys and queries), S grown until
    about budget_s of work."""
    import oracle
    oracle.build()
    with oracle.threads() as n:
        S, dt = _oracle_sample(w, budget_s)
    with oracle.threads(1):
        S1, dt1 = _oracle_sample(w, budget_s / 2)
    return {"value": round(S / dt, 1), "unit": "tokens/s", "cores": n, "kind": "oracle",
            "sample": f"first {S} of {w.T} tokens of the {w.name} workload (H={w.H}), "
                      f"keys and queries, {n} threads, {dt:.2f} s",
            "single_thread": {"value": round(S1 / dt1, 1), "unit": "tokens/s", "cores": 1,
                              "sample": f"first {S1} tokens, 1 thread, {dt1:.2f} s"}}


def run_ours(args):
    import torch
    from fp4_sparse_attention_fp4idx_gb300 import fp4idx as F
    from fp4_sparse_attention_fp4idx_gb300 import workloads as wl

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = init_dist(ws, "nccl")
    dev = torch.device("cuda", local)
    peak, peak_kind = measured_peak()
    flush = L2Flush(dev)

    w = wl.make(args.workload)
    D = upload(w, dev)
    sampler = ClockSampler(local) if rank == 0 else None
    r = time_device(F, w, D, args.mode, args.steps, args.warmup, flush, dist, sampler)
    step_sp = spread(r["step_ms"])
    step_ms = step_sp["median"]
    step_ms_all = max_over_ranks(step_ms, dist, dev)
    ab = algorithmic_bytes(w, args.mode)
    value = weak_scaling_value(ws, w.T, step_ms_all)

    # dominant kernel: the fused launch, or the query launch in separate mode
    kname = prepass_kernel_name(w.H)
    if args.mode == "fused":
        kbytes, kms = ab["fused"], step_ms
    else:
        kbytes, kms = ab["q_call"], float(np.median(r["q_ms"]))
    achieved = kbytes / (kms / 1e3) / 1e9
    tr = traffic_record(kname, w.name, args.mode)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                "kernel": kname, "algorithmic_bytes_per_launch": kbytes,
                "traffic": tr["dram_bytes_per_launch"] if tr else None}

    e2e_ms, h2d, d2h = time_e2e(F, w, D, args.mode, max(3, min(args.steps, 10)))
    e2e_ms_all = max_over_ranks(e2e_ms, dist, dev)

    extra = {}
    if rank == 0 and not args.no_extra:
        for name in ("prefill", "decode", "mtp"):
            if name == args.workload:
                continue
            wx = wl.make(name)
            Dx = upload(wx, dev)
            rx = time_device(F, wx, Dx, args.mode, 200, 5, flush)
            sp = spread(rx["step_ms"])
            ms = sp["median"]
            bx = algorithmic_bytes(wx, args.mode)["step"]
            extra[name] = {"T": wx.T, "H": wx.H, "ms_per_step": ms, "ms_spread": sp,
                           "tokens_per_s": round(wx.T / (ms / 1e3), 1),
                           "gbs": round(bx / (ms / 1e3) / 1e9, 1),
                           "frac_of_peak": round(bx / (ms / 1e3) / 1e9 / peak, 4)}
            del Dx

    scorer = variants = accuracy = None
    if rank == 0 and not args.no_extra and args.mode == "fused":
        variants = run_variants(F, w, D, dev, peak, flush)
    if rank == 0 and not args.no_extra:
        scorer = run_scorer(F, dev, peak, flush, 200)
        accuracy = run_accuracy(F, dev)

    base = cpu_baseline(w) if (rank == 0 and ws == 1 and not args.no_cpu) else None
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms_all, 5),
            "ms_per_step_spread": step_sp,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "T": w.T, "H": w.H, "head_dim": 128, "rope_dim": 64,
                       "rope_style": "neox" if w.rope_style == 0 else "interleaved",
                       "kv_blocks": w.num_blocks, "mode": args.mode,
                       "l2": "flushed before every timed step: write of a 2x L2 buffer, then a "
                             "read of another 2x L2 buffer (cleans the flush's dirty lines), "
                             "outside the step's CUDA events"},
            "gbs": round(ab["step"] / (step_ms_all / 1e3) / 1e9, 1),
            "frac_of_peak": round(ab["step"] / (step_ms_all / 1e3) / 1e9 / peak, 4),
            "algorithmic_bytes_per_step": ab["step"],
            "roofline": roofline,
            "e2e": {"value": round(weak_scaling_value(ws, w.T, e2e_ms_all), 1), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": round(e2e_ms_all, 4)},
            "gpu_launches": args.steps * (1 if args.mode == "fused" else 2),
            "clocks": r["clocks"],
            "cpu_baseline": base,
            "timed_wall_s": round(r["wall_s"], 4),
            "other_configs": extra,
            "variants": variants,
            "scorer": scorer,
            "accuracy": accuracy,
        }
        if args.mode != "fused":
            line["k_ms"] = round(float(np.median(r["k_ms"])), 5)
            line["q_ms"] = round(float(np.median(r["q_ms"])), 5)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ---------------------------------------------------------- reference arm
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from fp4_sparse_attention_fp4idx_gb300 import workloads as wl
    oracle.build()
    oracle.set_threads(oracle.threads_available())
    cores = oracle.get_threads()
    w = wl.make(args.workload)
    S = min(w.T, args.ref_tokens)
    cache = w.cache_init.copy()

    def step():
        oracle.k_norm_rope_pack_store(w.k[:S], w.gamma, w.eps, w.positions[:S], w.cos, w.sin,
                                      w.rope_style, w.slot_mapping[:S], cache)
        oracle.q_rope_pack_weights(w.q[:S], w.w[:S], w.positions[:S], w.cos, w.sin,
                                   w.rope_style)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = S / dt
    sample = (f"first {S} of {w.T} tokens of the {w.name} workload (H={w.H}) per step, "
              f"keys and queries, {cores} threads")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "H": w.H, "head_dim": 128, "rope_dim": 64,
                   "rope_style": "neox" if w.rope_style == 0 else "interleaved",
                   "kv_blocks": w.num_blocks, "mode": "oracle"},
        "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="large_prefill",
                    choices=["tiny", "decode", "prefill", "large_prefill", "mtp"])
    ap.add_argument("--mode", choices=["fused", "separate"], default="fused")
    ap.add_argument("--ref-tokens", type=int, default=4096,
                    help="tokens per step of the reference (oracle) arm")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-baseline leg")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

"""CPU-only checks of the boundary: the C-ABI library builds and loads, exports
every function include/fp4idx.h declares, and its host-side checks return the
documented status codes before anything touches CUDA.  Also checks that the
product path and the oracle never import each other."""
import ctypes
import os
import re
import shutil
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "fp4_sparse_attention_fp4idx_gb300")


@pytest.fixture(scope="module")
def F():
    from fp4_sparse_attention_fp4idx_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    from fp4_sparse_attention_fp4idx_gb300 import fp4idx
    return fp4idx


def test_exports_every_declared_symbol(F):
    names = F.declared_symbols()
    assert set(names) == {"fp4idx_k_norm_rope_pack_store", "fp4idx_q_rope_pack_weights",
                          "fp4idx_indexer_prepass", "fp4idx_paged_mqa_logits",
                          "fp4idx_k_norm_rope_pack_store_ex", "fp4idx_q_rope_pack_weights_ex",
                          "fp4idx_indexer_prepass_ex", "fp4idx_rope_fake_quant",
                          "fp4idx_mqa_logits_prefill", "fp4idx_default_weight_scale",
                          "fp4idx_test_withhold_next", "fp4idx_status_string",
                          "fp4idx_version", "fp4idx_indexer_prepass_host",
                          "fp4idx_host_staging_bytes", "fp4idx_indexer_prepass_host_static"}
    out = subprocess.run(["nm", "-D", "--defined-only", F.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (fp4idx_\w+)", out))
    assert set(names) <= exported
    for n in names:
        assert hasattr(F.lib(), n)


def test_library_is_built_for_sm103a(F):
    out = subprocess.run(["cuobjdump", "--list-elf", F.LIB_PATH], capture_output=True,
                         text=True)
    if out.returncode != 0:
        pytest.skip("cuobjdump unavailable")
    assert "sm_103a" in out.stdout


def test_status_strings_and_version(F):
    texts = [F.status_string(s) for s in range(7)]
    assert texts[0] == "ok" and len(set(texts)) == 7
    assert F.status_string(99) == "unknown status"
    assert F.version().startswith("fp4idx ") and "sm_103a" in F.version()


# Fake, aligned "device pointers": only ever passed together with a defect
# that the host checks reject, so nothing is dereferenced or launched.  As a
# second guard these tests never run where a CUDA device is visible (there
# the GPU suite checks the same status codes on real device memory).
A = [0x100000 * (i + 1) for i in range(20)]


@pytest.fixture(autouse=True)
def _no_visible_gpu(request):
    if "fake_ptr" in request.keywords:
        import torch
        if torch.cuda.is_available():
            pytest.skip("fake-pointer host-check tests run only where no GPU is visible")


def _k_args(**over):
    a = dict(k=A[0], k_stride=128, gamma=A[1], eps=1e-6, pos=A[2], cos=A[3], sin=A[4],
             max_pos=64, style=0, slots=A[5], cache=A[6], num_blocks=4, T=8, err=None,
             stream=None)
    a.update(over)
    return a


def _call_k(F, a):
    return F.lib().fp4idx_k_norm_rope_pack_store(
        a["k"], a["k_stride"], a["gamma"], a["eps"], a["pos"], a["cos"], a["sin"],
        a["max_pos"], a["style"], a["slots"], a["cache"], a["num_blocks"], a["T"], a["err"],
        a["stream"])


def _q_args(**over):
    a = dict(q=A[0], qts=64 * 128, qhs=128, w=A[7], wts=64, ws=0.125, pos=A[2], cos=A[3],
             sin=A[4], max_pos=64, style=1, qf=A[8], qs=A[9], wt=A[10], T=8, H=64, err=None,
             stream=None)
    a.update(over)
    return a


def _call_q(F, a):
    return F.lib().fp4idx_q_rope_pack_weights(
        a["q"], a["qts"], a["qhs"], a["w"], a["wts"], a["ws"], a["pos"], a["cos"], a["sin"],
        a["max_pos"], a["style"], a["qf"], a["qs"], a["wt"], a["T"], a["H"], a["err"],
        a["stream"])


def _call_fused(F, ka, qa):
    return F.lib().fp4idx_indexer_prepass(
        ka["k"], ka["k_stride"], ka["gamma"], ka["eps"], ka["slots"], ka["cache"],
        ka["num_blocks"], qa["q"], qa["qts"], qa["qhs"], qa["w"], qa["wts"], qa["ws"],
        qa["qf"], qa["qs"], qa["wt"], qa["H"], qa["pos"], qa["cos"], qa["sin"],
        qa["max_pos"], qa["style"], qa["T"], qa["err"], qa["stream"])


K_DEFECTS = [
    (dict(T=-1), "ERR_SHAPE"),
    (dict(k=None), "ERR_NULL"),
    (dict(gamma=None), "ERR_NULL"),
    (dict(pos=None), "ERR_NULL"),
    (dict(cos=None), "ERR_NULL"),
    (dict(sin=None), "ERR_NULL"),
    (dict(slots=None), "ERR_NULL"),
    (dict(cache=None), "ERR_NULL"),
    (dict(max_pos=0), "ERR_SHAPE"),
    (dict(num_blocks=0), "ERR_SHAPE"),
    (dict(num_blocks=1 << 62), "ERR_SHAPE"),
    (dict(style=2), "ERR_ARG"),
    (dict(style=-1), "ERR_ARG"),
    (dict(eps=0.0), "ERR_ARG"),
    (dict(eps=-1e-6), "ERR_ARG"),
    (dict(eps=float("nan")), "ERR_ARG"),
    (dict(eps=float("inf")), "ERR_ARG"),
    (dict(k=A[0] + 8), "ERR_ALIGN"),
    (dict(k_stride=130), "ERR_ALIGN"),
    (dict(gamma=A[1] + 2), "ERR_ALIGN"),
    (dict(pos=A[2] + 4), "ERR_ALIGN"),
    (dict(cos=A[3] + 4), "ERR_ALIGN"),
    (dict(slots=A[5] + 4), "ERR_ALIGN"),
    (dict(cache=A[6] + 4), "ERR_ALIGN"),
    (dict(err=A[11] + 2), "ERR_ALIGN"),
]

Q_DEFECTS = [
    (dict(T=-3), "ERR_SHAPE"),
    (dict(q=None), "ERR_NULL"),
    (dict(w=None), "ERR_NULL"),
    (dict(qf=None), "ERR_NULL"),
    (dict(qs=None), "ERR_NULL"),
    (dict(wt=None), "ERR_NULL"),
    (dict(pos=None), "ERR_NULL"),
    (dict(H=0), "ERR_SHAPE"),
    (dict(H=1 << 60), "ERR_SHAPE"),
    (dict(max_pos=-5), "ERR_SHAPE"),
    (dict(style=7), "ERR_ARG"),
    (dict(ws=float("inf")), "ERR_ARG"),
    (dict(ws=float("nan")), "ERR_ARG"),
    (dict(q=A[0] + 2), "ERR_ALIGN"),
    (dict(qts=64 * 128 + 4), "ERR_ALIGN"),
    (dict(qhs=132), "ERR_ALIGN"),
    (dict(w=A[7] + 1), "ERR_ALIGN"),
    (dict(qf=A[8] + 4), "ERR_ALIGN"),
    (dict(qs=A[9] + 2), "ERR_ALIGN"),
    (dict(wt=A[10] + 2), "ERR_ALIGN"),
    (dict(sin=A[4] + 8), "ERR_ALIGN"),
]


def _ids(defects):
    return [f"{list(o)[0]}={list(o.values())[0]}" for o, _ in defects]


# Arguments the fused call takes from the key side only; everything else
# (positions, tables, max_pos, rope_style, T) comes from the query side.
_KEY_ONLY = {"k", "k_stride", "gamma", "eps", "slots", "cache", "num_blocks", "err"}
FUSED_K_DEFECTS = [d for d in K_DEFECTS if set(d[0]) <= _KEY_ONLY and "err" not in d[0]]
FUSED_Q_DEFECTS = Q_DEFECTS


@pytest.mark.fake_ptr
@pytest.mark.parametrize("over,code", K_DEFECTS, ids=_ids(K_DEFECTS))
def test_key_host_checks(F, over, code):
    assert _call_k(F, _k_args(**over)) == getattr(F, code)


@pytest.mark.fake_ptr
@pytest.mark.parametrize("over,code", Q_DEFECTS, ids=_ids(Q_DEFECTS))
def test_query_host_checks(F, over, code):
    assert _call_q(F, _q_args(**over)) == getattr(F, code)


@pytest.mark.fake_ptr
@pytest.mark.parametrize("over,code", FUSED_K_DEFECTS, ids=_ids(FUSED_K_DEFECTS))
def test_fused_host_checks_keys(F, over, code):
    assert _call_fused(F, _k_args(**over), _q_args(style=0)) == getattr(F, code)


@pytest.mark.fake_ptr
@pytest.mark.parametrize("over,code", FUSED_Q_DEFECTS, ids=_ids(FUSED_Q_DEFECTS))
def test_fused_host_checks_queries(F, over, code):
    assert _call_fused(F, _k_args(), _q_args(**over)) == getattr(F, code)


def _s_args(**over):
    a = dict(qf=A[12], qs=A[13], w=A[14], cache=A[6], nb=16, bt=A[15], bts=8, ctx=A[16],
             out=A[17], os=512, batch=4, next_n=1, H=32, max_ctx=500, err=None, stream=None)
    a.update(over)
    return a


def _call_s(F, a):
    return F.lib().fp4idx_paged_mqa_logits(
        a["qf"], a["qs"], a["w"], a["cache"], a["nb"], a["bt"], a["bts"], a["ctx"], a["out"],
        a["os"], a["batch"], a["next_n"], a["H"], a["max_ctx"], a["err"], a["stream"])


S_DEFECTS = [
    (dict(batch=-1), "ERR_SHAPE"),
    (dict(max_ctx=-1), "ERR_SHAPE"),
    (dict(qf=None), "ERR_NULL"),
    (dict(qs=None), "ERR_NULL"),
    (dict(w=None), "ERR_NULL"),
    (dict(cache=None), "ERR_NULL"),
    (dict(bt=None), "ERR_NULL"),
    (dict(ctx=None), "ERR_NULL"),
    (dict(out=None), "ERR_NULL"),
    (dict(next_n=0), "ERR_SHAPE"),
    (dict(H=16), "ERR_SHAPE"),
    (dict(H=48), "ERR_SHAPE"),
    (dict(H=160), "ERR_SHAPE"),
    (dict(H=288), "ERR_SHAPE"),
    (dict(nb=0), "ERR_SHAPE"),
    (dict(nb=1 << 40), "ERR_SHAPE"),
    (dict(max_ctx=1 << 30), "ERR_SHAPE"),
    (dict(os=499), "ERR_SHAPE"),
    (dict(bts=7), "ERR_SHAPE"),
    (dict(qf=A[12] + 4), "ERR_ALIGN"),
    (dict(qs=A[13] + 2), "ERR_ALIGN"),
    (dict(w=A[14] + 2), "ERR_ALIGN"),
    (dict(cache=A[6] + 8), "ERR_ALIGN"),
    (dict(bt=A[15] + 2), "ERR_ALIGN"),
    (dict(ctx=A[16] + 1), "ERR_ALIGN"),
    (dict(out=A[17] + 2), "ERR_ALIGN"),
    (dict(err=A[11] + 2), "ERR_ALIGN"),
]


@pytest.mark.fake_ptr
@pytest.mark.parametrize("over,code", S_DEFECTS, ids=_ids(S_DEFECTS))
def test_scorer_host_checks(F, over, code):
    assert _call_s(F, _s_args(**over)) == getattr(F, code)


def _p_args(**over):
    a = dict(qf=A[12], qs=A[13], w=A[14], cache=A[6], nb=16, nk=1000, ks=A[15], ke=A[16],
             out=A[17], os=1000, T=7, H=64, err=None, stream=None)
    a.update(over)
    return a


def _call_p(F, a):
    return F.lib().fp4idx_mqa_logits_prefill(
        a["qf"], a["qs"], a["w"], a["cache"], a["nb"], a["nk"], a["ks"], a["ke"], a["out"],
        a["os"], a["T"], a["H"], a["err"], a["stream"])


P_DEFECTS = [
    (dict(T=-1), "ERR_SHAPE"),
    (dict(nk=-1), "ERR_SHAPE"),
    (dict(qf=None), "ERR_NULL"),
    (dict(ks=None), "ERR_NULL"),
    (dict(ke=None), "ERR_NULL"),
    (dict(out=None), "ERR_NULL"),
    (dict(H=16), "ERR_SHAPE"),
    (dict(H=80), "ERR_SHAPE"),
    (dict(H=288), "ERR_SHAPE"),
    (dict(H=160), "ERR_SHAPE"),
    (dict(nb=0), "ERR_SHAPE"),
    (dict(nk=16 * 64 + 1), "ERR_SHAPE"),
    (dict(os=999), "ERR_SHAPE"),
    (dict(qf=A[12] + 4), "ERR_ALIGN"),
    (dict(cache=A[6] + 8), "ERR_ALIGN"),
    (dict(ks=A[15] + 2), "ERR_ALIGN"),
    (dict(out=A[17] + 2), "ERR_ALIGN"),
]


@pytest.mark.fake_ptr
@pytest.mark.parametrize("over,code", P_DEFECTS, ids=_ids(P_DEFECTS))
def test_prefill_scorer_host_checks(F, over, code):
    assert _call_p(F, _p_args(**over)) == getattr(F, code)


def test_prefill_scorer_empty_is_a_no_op(F):
    assert _call_p(F, _p_args(T=0)) == F.OK and _call_p(F, _p_args(nk=0)) == F.OK


@pytest.mark.fake_ptr
@pytest.mark.parametrize("ratio,had,mode", [(3, 0, 0), (0, 0, 0), (8, 0, 0), (1, 2, 0),
                                            (2, -1, 0), (1, 0, 2), (1, 0, -1)])
def test_option_host_checks(F, ratio, had, mode):
    """A bad options block is rejected on the host (ERR_ARG) by all three
    variant entry points."""
    import ctypes
    opts = ctypes.cast(ctypes.pointer(F.Options(ratio, had, mode)), ctypes.c_void_p)
    ka, qa = _k_args(), _q_args(style=0)
    assert F.lib().fp4idx_k_norm_rope_pack_store_ex(
        ka["k"], ka["k_stride"], ka["gamma"], ka["eps"], ka["pos"], ka["cos"], ka["sin"],
        ka["max_pos"], ka["style"], ka["slots"], ka["cache"], ka["num_blocks"], ka["T"], opts,
        None, None) == F.ERR_ARG
    assert F.lib().fp4idx_q_rope_pack_weights_ex(
        qa["q"], qa["qts"], qa["qhs"], qa["w"], qa["wts"], qa["ws"], qa["pos"], qa["cos"],
        qa["sin"], qa["max_pos"], qa["style"], qa["qf"], qa["qs"], qa["wt"], qa["T"], qa["H"],
        opts, None, None) == F.ERR_ARG
    assert F.lib().fp4idx_indexer_prepass_ex(
        ka["k"], ka["k_stride"], ka["gamma"], ka["eps"], ka["slots"], ka["cache"],
        ka["num_blocks"], qa["q"], qa["qts"], qa["qhs"], qa["w"], qa["wts"], qa["ws"],
        qa["qf"], qa["qs"], qa["wt"], qa["H"], qa["pos"], qa["cos"], qa["sin"],
        qa["max_pos"], qa["style"], qa["T"], opts, None, None) == F.ERR_ARG


FQ_DEFECTS = [
    (dict(n=-1), "ERR_SHAPE"),
    (dict(x=None), "ERR_NULL"),
    (dict(out=None), "ERR_NULL"),
    (dict(pos=None), "ERR_NULL"),
    (dict(per=0), "ERR_SHAPE"),
    (dict(stride=64), "ERR_SHAPE"),
    (dict(n=1 << 31), "ERR_SHAPE"),
    (dict(mode=2), "ERR_ARG"),
    (dict(style=3), "ERR_ARG"),
    (dict(x=A[0] + 8), "ERR_ALIGN"),
    (dict(stride=132), "ERR_ALIGN"),
    (dict(out=A[18] + 2), "ERR_ALIGN"),
    (dict(max_pos=0), "ERR_SHAPE"),
]


@pytest.mark.fake_ptr
@pytest.mark.parametrize("over,code", FQ_DEFECTS, ids=_ids(FQ_DEFECTS))
def test_fake_quant_host_checks(F, over, code):
    a = dict(x=A[0], stride=128, per=1, pos=A[2], cos=A[3], sin=A[4], max_pos=64, style=0,
             mode=1, out=A[18], n=64, err=None, stream=None)
    a.update(over)
    assert F.lib().fp4idx_rope_fake_quant(
        a["x"], a["stride"], a["per"], a["pos"], a["cos"], a["sin"], a["max_pos"], a["style"],
        a["mode"], a["out"], a["n"], a["err"], a["stream"]) == getattr(F, code)


# fp4idx_indexer_prepass_host: k, q, w, slots, positions and the outputs are
# host pointers, the rest device pointers; none is touched before a defect.
def _h_args(**over):
    a = dict(k=A[0], slots=A[5], gamma=A[1], eps=1e-6, cache=A[6], num_blocks=4, q=A[7],
             w=A[8], H=32, ws=0.125, qf=A[9], qs=A[10], wt=A[11], pos=A[2], cos=A[3],
             sin=A[4], max_pos=64, style=0, T=100, chunk=32, staging=A[12], err=None,
             stream=None)
    a.update(over)
    return a


def _call_h(F, a):
    return F.lib().fp4idx_indexer_prepass_host(
        a["k"], a["slots"], a["gamma"], a["eps"], a["cache"], a["num_blocks"], a["q"], a["w"],
        a["H"], a["ws"], a["qf"], a["qs"], a["wt"], a["pos"], a["cos"], a["sin"], a["max_pos"],
        a["style"], a["T"], a["chunk"], a["staging"], a["err"], a["stream"])


H_DEFECTS = [
    (dict(T=-1), "ERR_SHAPE"),
    (dict(H=0), "ERR_SHAPE"),
    (dict(chunk=0), "ERR_SHAPE"),
    (dict(chunk=1 << 30), "ERR_SHAPE"),
    (dict(H=1 << 20, chunk=1 << 10), "ERR_SHAPE"),
    (dict(max_pos=0), "ERR_SHAPE"),
    (dict(num_blocks=0), "ERR_SHAPE"),
    *[(dict([(n, None)]), "ERR_NULL") for n in ("k", "slots", "gamma", "cache", "q", "w",
                                                 "qf", "qs", "wt", "pos", "cos", "sin",
                                                 "staging")],
    (dict(staging=A[12] + 16), "ERR_ALIGN"),
    (dict(gamma=A[1] + 2), "ERR_ALIGN"),
    (dict(cos=A[3] + 4), "ERR_ALIGN"),
    (dict(cache=A[6] + 4), "ERR_ALIGN"),
    (dict(err=A[13] + 2), "ERR_ALIGN"),
    (dict(eps=0.0), "ERR_ARG"),
    (dict(style=3), "ERR_ARG"),
    (dict(ws=float("nan")), "ERR_ARG"),
]


@pytest.mark.fake_ptr
@pytest.mark.parametrize("over,code", H_DEFECTS, ids=_ids(H_DEFECTS))
def test_host_pipeline_host_checks(F, over, code):
    assert _call_h(F, _h_args(**over)) == getattr(F, code)


def test_host_staging_bytes(F):
    L = F.lib()
    # two slots, each the chunk's inputs and query outputs in 256-byte
    # aligned pieces: q 64*32*256, k 64*256, w 64*32*2, positions and slots
    # 64*8 each, q_fp4 64*32*64, q_scale and weights 64*32*4 each
    assert L.fp4idx_host_staging_bytes(64, 32) == 2 * (524288 + 16384 + 4096 + 512 + 512
                                                      + 131072 + 8192 + 8192)
    # a ragged size rounds every piece up to 256 bytes
    assert L.fp4idx_host_staging_bytes(1, 1) == 2 * 8 * 256
    for c, h in ((0, 32), (32, 0), (-1, 1), (1 << 30, 1), (1 << 15, 1 << 15)):
        assert L.fp4idx_host_staging_bytes(c, h) == 0


def _call_hs(F, a):
    return F.lib().fp4idx_indexer_prepass_host_static(
        a["k"], a["slots"], a["gamma"], a["eps"], a["cache"], a["num_blocks"], a["q"], a["w"],
        a["H"], a["ws"], a["qf"], a["qs"], a["wt"], a["pos"], a["cos"], a["sin"], a["max_pos"],
        a["style"], a["T"], a["chunk"], a["err"], a["stream"])


@pytest.mark.fake_ptr
@pytest.mark.parametrize("over,code", [
    (dict(T=-1), "ERR_SHAPE"), (dict(H=0), "ERR_SHAPE"), (dict(chunk=0), "ERR_SHAPE"),
    (dict(chunk=1 << 30), "ERR_SHAPE"),
    (dict(chunk=4096, H=64), "ERR_SCRATCH"),       # 168 MB of staging
    (dict(chunk=1569, H=64), "ERR_SCRATCH"),       # just past the buffer (1568 fit)
    (dict(chunk=100000, H=1), "ERR_SCRATCH"),
    (dict(T=0, k=None, q=None), "OK"),
], ids=["T", "H", "chunk0", "chunk_overflow", "4096x64", "1569x64", "100000x1", "empty"])
def test_static_staging_host_checks(F, over, code):
    """The static-staging call rejects a request its buffer cannot hold
    before it looks the buffer up or enqueues anything."""
    assert _call_hs(F, _h_args(**over)) == getattr(F, code)


def test_static_staging_bound(F):
    """The header's sufficient condition for a chunk to fit the static
    buffer, c * (660 H + 544) + 4096 <= FP4IDX_STATIC_STAGING_BYTES, holds
    against the library's staging size, and its example fits."""
    text = open(F.HEADER_PATH).read()
    assert "FP4IDX_STATIC_STAGING_BYTES = 64 << 20" in text
    L = F.lib()
    for c, h in ((1536, 64), (3072, 32), (1, 1), (777, 17), (12000, 8)):
        exact = L.fp4idx_host_staging_bytes(c, h)
        assert c * (660 * h + 544) <= exact <= c * (660 * h + 544) + 4096
    assert L.fp4idx_host_staging_bytes(1536, 64) <= F.STATIC_STAGING_BYTES
    assert L.fp4idx_host_staging_bytes(1568, 64) <= F.STATIC_STAGING_BYTES
    assert L.fp4idx_host_staging_bytes(1569, 64) > F.STATIC_STAGING_BYTES


@pytest.mark.fake_ptr
def test_zero_tokens_is_ok_without_touching_cuda(F):
    # All pointers NULL, T == 0: returns OK before any check or CUDA call.
    assert _call_k(F, _k_args(T=0, k=None, gamma=None, cache=None)) == F.OK
    assert _call_q(F, _q_args(T=0, q=None, w=None)) == F.OK
    assert _call_fused(F, _k_args(T=0), _q_args(T=0)) == F.OK
    assert _call_s(F, _s_args(batch=0, qf=None, cache=None)) == F.OK
    assert _call_s(F, _s_args(max_ctx=0, out=None)) == F.OK
    assert _call_h(F, _h_args(T=0, k=None, q=None, staging=None)) == F.OK


def test_binding_fails_loudly_without_the_library(tmp_path):
    """No CPU fallback: importing the binding without libfp4idx.so raises."""
    pkg = tmp_path / "fp4_sparse_attention_fp4idx_gb300"
    shutil.copytree(PKG, pkg, ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    r = subprocess.run([sys.executable, "-c",
                        "import fp4_sparse_attention_fp4idx_gb300.fp4idx"],
                       cwd=tmp_path, capture_output=True, text=True)
    assert r.returncode != 0 and "ImportError" in r.stderr and "no CPU fallback" in r.stderr


def _py_sources(d):
    for dp, _, fs in os.walk(d):
        for f in fs:
            if f.endswith((".py", ".cu", ".h", ".c")):
                yield os.path.join(dp, f)


def test_product_and_oracle_are_independent():
    """The package never imports the oracle, and the oracle never imports the
    package (they share only the seeded workload generator via the tests)."""
    for p in _py_sources(PKG):
        text = open(p).read()
        assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), p
        assert "fp4idx_oracle" not in text, p
    for p in _py_sources(os.path.join(ROOT, "oracle")):
        text = open(p).read()
        assert not re.search(r"^\s*(import|from)\s+fp4_sparse_attention_fp4idx_gb300\b",
                             text, re.M), p
        assert not re.search(r"#\s*include\s*[<\"]fp4idx\.h", text), p


def test_default_weight_scale_closed_form(F):
    """The library's head-weight scale is H^-1/2 * 128^-1/2 rounded once to
    fp32 (aiter PR 5484, API; sglang PR 39656, Summary); exact powers of two
    where H * 128 is a power of four."""
    import numpy as np
    from fractions import Fraction
    assert F.default_weight_scale(32) == 1.0 / 64 and F.default_weight_scale(128) == 1.0 / 128
    for H in (1, 8, 12, 17, 32, 48, 64, 96, 128, 1000):
        got = F.default_weight_scale(H)
        want = np.float32(1.0 / np.sqrt(np.float64(H) * 128.0))
        assert got == float(want), H
        # within half an fp32 ulp of the exact value
        exact = 1.0 / (H * 128) ** 0.5
        assert abs(Fraction(got) - Fraction(exact)) <= Fraction(float(np.spacing(want))) / 2 * (1 + 1e-9)
    assert F.default_weight_scale(0) == 0.0


def test_withhold_hook_argument_checks(F):
    """The testing hook only arms itself for a known kernel and a
    non-negative index (host-side, no launch); index 2^40 withholds nothing
    (it is past any CTA's work) and is taken by the next launch."""
    L = F.lib()
    assert L.fp4idx_test_withhold_next(7, 0) == F.ERR_ARG
    assert L.fp4idx_test_withhold_next(F.TEST_SCORER, -1) == F.ERR_ARG
    assert L.fp4idx_test_withhold_next(F.TEST_PREPASS, 1 << 40) == F.OK
    assert L.fp4idx_test_withhold_next(F.TEST_SCORER, 1 << 40) == F.OK

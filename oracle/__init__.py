"""Plain scalar CPU oracle of the fused FP4 indexer pre-pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference legs of ``bench.py`` may import this package.
The product path (``fp4_sparse_attention_fp4idx_gb300``) never does, and this
package never imports the product.

The arithmetic lives in ``fp4idx_oracle.c`` (plain C, compiled without FP
contraction); this module only builds it with gcc and marshals numpy arrays.
bf16 arrays are carried as ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp4idx_oracle.c")
_LIB = os.path.join(_HERE, "libfp4idx_oracle.so")

HEAD_DIM = 128
PAYLOAD_BYTES = 64
EXP_BYTES = 4
KV_BLOCK = 64
PAGE_BYTES = KV_BLOCK * (PAYLOAD_BYTES + EXP_BYTES)
FP8_PAGE_BYTES = KV_BLOCK * (HEAD_DIM + 4)
ROPE_NEOX = 0
ROPE_INTERLEAVED = 1


_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fno-strict-aliasing",
           "-shared", "-fPIC"]


def _gcc(src: str, out: str) -> None:
    """gcc with OpenMP (token-parallel loops) when the toolchain has it, else
    without (the pragmas are then ignored and the oracle runs one thread)."""
    try:
        subprocess.run(["gcc", *_CFLAGS, "-fopenmp", "-o", out, src, "-lm"], check=True,
                       stderr=subprocess.DEVNULL)
    except subprocess.CalledProcessError:
        subprocess.run(["gcc", *_CFLAGS, "-Wno-unknown-pragmas", "-o", out, src, "-lm"],
                       check=True)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FP contraction, no fast-math)."""
    hdr = os.path.join(_HERE, "fp4idx_oracle.h")
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= max(os.path.getmtime(_SRC), os.path.getmtime(hdr))):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    _gcc(_SRC, tmp)
    os.replace(tmp, _LIB)
    return _LIB


def _bind(L: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    L.oracle_f32_to_bf16.restype = ctypes.c_uint16
    L.oracle_rmsnorm_row.argtypes = [P, P, ctypes.c_float, P]
    L.oracle_rmsnorm_row.restype = None
    L.oracle_rope_row.argtypes = [P, P, P, ctypes.c_int]
    L.oracle_rope_row.restype = None
    L.oracle_quant_group.argtypes = [P, ctypes.c_float, P]
    L.oracle_quant_group.restype = ctypes.c_int
    L.oracle_quant_group_floors.argtypes = [P, ctypes.c_float, ctypes.c_float, P]
    L.oracle_quant_group_floors.restype = ctypes.c_int
    L.oracle_quant_pack_row_floors.argtypes = [P, ctypes.c_float, ctypes.c_float,
                                               ctypes.c_float, ctypes.c_float, P, P, P, P, P]
    L.oracle_quant_pack_row_floors.restype = None
    L.oracle_dequant.argtypes = [ctypes.c_uint8, ctypes.c_int]
    L.oracle_dequant.restype = ctypes.c_float
    L.oracle_quant_pack_row.argtypes = [P, P, P, P, P, P]
    L.oracle_quant_pack_row.restype = None
    L.oracle_k_norm_rope_pack_store.argtypes = [
        P, P, ctypes.c_float, P, P, P, i64, ctypes.c_int, P, P, i64, i64]
    L.oracle_k_norm_rope_pack_store.restype = ctypes.c_int
    L.oracle_q_rope_pack_weights.argtypes = [
        P, P, P, P, P, i64, ctypes.c_int, P, P, P, i64, i64]
    L.oracle_q_rope_pack_weights.restype = ctypes.c_int
    L.oracle_hadamard_row.argtypes = [P]
    L.oracle_hadamard_row.restype = None
    L.oracle_k_norm_rope_pack_store_ex.argtypes = [
        P, P, ctypes.c_float, P, P, P, i64, ctypes.c_int, P, P, i64, i64, ctypes.c_int,
        ctypes.c_int]
    L.oracle_k_norm_rope_pack_store_ex.restype = ctypes.c_int
    L.oracle_q_rope_pack_weights_ex.argtypes = [
        P, P, P, P, P, i64, ctypes.c_int, P, P, P, i64, i64, ctypes.c_int]
    L.oracle_q_rope_pack_weights_ex.restype = ctypes.c_int
    L.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_to_f32.restype = ctypes.c_float
    L.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
    L.oracle_f32_to_e4m3.restype = ctypes.c_uint8
    L.oracle_fp8_quant_row.argtypes = [P, P]
    L.oracle_fp8_quant_row.restype = ctypes.c_int
    L.oracle_k_norm_rope_fp8_store.argtypes = [
        P, P, ctypes.c_float, P, P, P, i64, ctypes.c_int, P, P, i64, i64, ctypes.c_int,
        ctypes.c_int]
    L.oracle_k_norm_rope_fp8_store.restype = ctypes.c_int
    L.oracle_q_rope_fp8_weights.argtypes = [
        P, P, P, P, P, i64, ctypes.c_int, P, P, i64, i64, ctypes.c_int]
    L.oracle_q_rope_fp8_weights.restype = ctypes.c_int
    L.oracle_fake_quant_row.argtypes = [P, ctypes.c_int, P]
    L.oracle_fake_quant_row.restype = None
    L.oracle_rope_fake_quant.argtypes = [P, i64, P, P, P, i64, ctypes.c_int, ctypes.c_int, P, i64]
    L.oracle_rope_fake_quant.restype = ctypes.c_int
    L.oracle_paged_mqa_logits.argtypes = [
        P, P, P, P, i64, P, i64, P, P, i64, i64, i64, i64, i64]
    L.oracle_paged_mqa_logits.restype = ctypes.c_int
    L.oracle_mqa_logits_prefill.argtypes = [P, P, P, P, i64, P, P, P, i64, i64, i64]
    L.oracle_mqa_logits_prefill.restype = ctypes.c_int
    L.oracle_set_threads.argtypes = [ctypes.c_int]
    L.oracle_set_threads.restype = None
    L.oracle_get_threads.argtypes = []
    L.oracle_get_threads.restype = ctypes.c_int
    L.oracle_threads_available.argtypes = []
    L.oracle_threads_available.restype = ctypes.c_int
    return L


_lib = None
_active = None  # set by use_variant(): a planted-mistake build for mutation tests


def lib() -> ctypes.CDLL:
    global _lib
    if _active is not None:
        return _active
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def compile_variant(source_text: str, workdir: str) -> ctypes.CDLL:
    """Compile a modified copy of the oracle's C source (used by the tests to
    plant a mistake and check that the pins catch it)."""
    import shutil
    src = os.path.join(workdir, "fp4idx_oracle.c")
    shutil.copy(os.path.join(_HERE, "fp4idx_oracle.h"), workdir)
    with open(src, "w") as f:
        f.write(source_text)
    so = os.path.join(workdir, f"libvariant{abs(hash(source_text))}.so")
    _gcc(src, so)
    return _bind(ctypes.CDLL(so))


class use_variant:
    """Context manager: route every oracle call to the given library."""

    def __init__(self, L):
        self.L = L

    def __enter__(self):
        global _active
        self.prev, _active = _active, self.L
        return self.L

    def __exit__(self, *exc):
        global _active
        _active = self.prev
        return False


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- single steps
def f32_to_bf16(x: float) -> int:
    return int(lib().oracle_f32_to_bf16(ctypes.c_float(x)))


def rmsnorm_row(x_bits, gamma_bits, eps: float) -> np.ndarray:
    x = _c(x_bits, np.uint16)
    g = _c(gamma_bits, np.uint16)
    assert x.shape == (HEAD_DIM,) and g.shape == (HEAD_DIM,)
    y = np.empty(HEAD_DIM, np.uint16)
    lib().oracle_rmsnorm_row(_p(x), _p(g), ctypes.c_float(eps), _p(y))
    return y


def rope_row(y_bits, cos_row, sin_row, rope_style: int) -> np.ndarray:
    y = _c(y_bits, np.uint16).copy()
    c = _c(cos_row, np.float32)
    s = _c(sin_row, np.float32)
    assert y.shape == (HEAD_DIM,) and c.shape == (32,) and s.shape == (32,)
    lib().oracle_rope_row(_p(y), _p(c), _p(s), int(rope_style))
    return y


def quant_group(z, floor: float = 2.0 ** -126):
    """Returns (nibbles uint8[32], exponent)."""
    z = _c(z, np.float32)
    assert z.shape == (32,)
    n = np.empty(32, np.uint8)
    e = lib().oracle_quant_group(_p(z), ctypes.c_float(floor), _p(n))
    return n, int(e)


def quant_group_floors(z, amax_floor: float, quot_floor: float):
    """(nibbles uint8[32], exponent) with a floor on the amax (before the
    division by 6) and one on the quotient (after it); 0 = no floor."""
    z = _c(z, np.float32)
    assert z.shape == (32,)
    n = np.empty(32, np.uint8)
    e = lib().oracle_quant_group_floors(_p(z), ctypes.c_float(amax_floor),
                                        ctypes.c_float(quot_floor), _p(n))
    return n, int(e)


def quant_pack_row_floors(row_bits, s1_amax: float, s1_quot: float, s2_amax: float,
                          s2_quot: float):
    """quant_pack_row with explicit floors for both stages."""
    r = _c(row_bits, np.uint16)
    assert r.shape == (HEAD_DIM,)
    payload = np.empty(PAYLOAD_BYTES, np.uint8)
    ex = np.empty(EXP_BYTES, np.uint8)
    e1 = np.empty(4, np.int32)
    e2 = np.empty(4, np.int32)
    n1 = np.empty(HEAD_DIM, np.uint8)
    lib().oracle_quant_pack_row_floors(_p(r), ctypes.c_float(s1_amax), ctypes.c_float(s1_quot),
                                       ctypes.c_float(s2_amax), ctypes.c_float(s2_quot),
                                       _p(payload), _p(ex), _p(e1), _p(e2), _p(n1))
    return dict(payload=payload, exp=ex, e1=e1, e2=e2, n1=n1)


def set_threads(n: int) -> None:
    """Host threads for the oracle's token / row loops (1 = single-threaded)."""
    lib().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(lib().oracle_get_threads())


def threads_available() -> int:
    """Cores the oracle can use (1 if it was built without OpenMP)."""
    return int(lib().oracle_threads_available())


class threads:
    """Context manager: run the oracle on n host threads (default: all)."""

    def __init__(self, n: int | None = None):
        self.n = n

    def __enter__(self):
        self.prev = get_threads()
        set_threads(self.n or threads_available())
        return get_threads()

    def __exit__(self, *exc):
        set_threads(self.prev)
        return False


def dequant(nibble: int, e: int) -> float:
    return float(lib().oracle_dequant(ctypes.c_uint8(nibble), int(e)))


def quant_pack_row(row_bits):
    """Returns dict(payload[64], exp[4], e1[4], e2[4], n1[128])."""
    r = _c(row_bits, np.uint16)
    assert r.shape == (HEAD_DIM,)
    payload = np.empty(PAYLOAD_BYTES, np.uint8)
    ex = np.empty(EXP_BYTES, np.uint8)
    e1 = np.empty(4, np.int32)
    e2 = np.empty(4, np.int32)
    n1 = np.empty(HEAD_DIM, np.uint8)
    lib().oracle_quant_pack_row(_p(r), _p(payload), _p(ex), _p(e1), _p(e2), _p(n1))
    return dict(payload=payload, exp=ex, e1=e1, e2=e2, n1=n1)


# ------------------------------------------------------------------ full ops
def hadamard_row(y_bits) -> np.ndarray:
    """Normalised 128-point Walsh-Hadamard rotation of a bf16 row (bits)."""
    y = _c(y_bits, np.uint16).copy()
    assert y.shape == (HEAD_DIM,)
    lib().oracle_hadamard_row(_p(y))
    return y


def k_norm_rope_pack_store(k, gamma, eps, positions, cos_cache, sin_cache,
                           rope_style, slot_mapping, kv_cache, compress_ratio: int = 1,
                           hadamard: bool = False) -> int:
    """kv_cache (uint8 [num_blocks, 4352]) is updated in place."""
    k = _c(k, np.uint16)
    T = k.shape[0]
    assert k.shape == (T, HEAD_DIM)
    g = _c(gamma, np.uint16)
    pos = _c(positions, np.int64)
    cs = _c(cos_cache, np.float32)
    sn = _c(sin_cache, np.float32)
    sl = _c(slot_mapping, np.int64)
    assert kv_cache.dtype == np.uint8 and kv_cache.flags.c_contiguous
    assert kv_cache.shape[1:] == (PAGE_BYTES,)
    assert pos.shape == (T,) and sl.shape == (T,) and cs.shape == sn.shape
    return int(lib().oracle_k_norm_rope_pack_store_ex(
        _p(k), _p(g), ctypes.c_float(eps), _p(pos), _p(cs), _p(sn), cs.shape[0],
        int(rope_style), _p(sl), _p(kv_cache), kv_cache.shape[0], T, int(compress_ratio),
        int(bool(hadamard))))


def q_rope_pack_weights(q, w, positions, cos_cache, sin_cache, rope_style,
                        out=None, hadamard: bool = False):
    """Returns (q_fp4 [T,H,64] u8, q_scale [T,H,4] u8, weights [T,H] f32, status)."""
    q = _c(q, np.uint16)
    T, H, D = q.shape
    assert D == HEAD_DIM
    w = _c(w, np.uint16)
    assert w.shape == (T, H)
    pos = _c(positions, np.int64)
    cs = _c(cos_cache, np.float32)
    sn = _c(sin_cache, np.float32)
    if out is None:
        out = (np.zeros((T, H, PAYLOAD_BYTES), np.uint8),
               np.zeros((T, H, EXP_BYTES), np.uint8),
               np.zeros((T, H), np.float32))
    qf, qs, wt = out
    st = lib().oracle_q_rope_pack_weights_ex(
        _p(q), _p(w), _p(pos), _p(cs), _p(sn), cs.shape[0], int(rope_style),
        _p(qf), _p(qs), _p(wt), T, H, int(bool(hadamard)))
    return qf, qs, wt, int(st)


def e4m3_to_f32(c: int) -> float:
    return float(lib().oracle_e4m3_to_f32(int(c)))


def f32_to_e4m3(v: float) -> int:
    return int(lib().oracle_f32_to_e4m3(float(v)))


def fp8_quant_row(row_bits):
    """(codes uint8 [128], biased exponent e of the row scale 2^(e-127))."""
    r = _c(row_bits, np.uint16)
    assert r.shape == (HEAD_DIM,)
    codes = np.zeros(HEAD_DIM, np.uint8)
    e = lib().oracle_fp8_quant_row(_p(r), _p(codes))
    return codes, int(e)


def k_norm_rope_fp8_store(k, gamma, eps, positions, cos_cache, sin_cache, rope_style,
                          slot_mapping, kv_cache, compress_ratio: int = 1,
                          hadamard: bool = False) -> int:
    """FP8 mode; kv_cache (uint8 [num_blocks, 8448]) is updated in place."""
    k = _c(k, np.uint16)
    T = k.shape[0]
    assert k.shape == (T, HEAD_DIM)
    g = _c(gamma, np.uint16)
    pos = _c(positions, np.int64)
    cs = _c(cos_cache, np.float32)
    sn = _c(sin_cache, np.float32)
    sl = _c(slot_mapping, np.int64)
    assert kv_cache.dtype == np.uint8 and kv_cache.flags.c_contiguous
    assert kv_cache.shape[1:] == (FP8_PAGE_BYTES,)
    return int(lib().oracle_k_norm_rope_fp8_store(
        _p(k), _p(g), ctypes.c_float(eps), _p(pos), _p(cs), _p(sn), cs.shape[0],
        int(rope_style), _p(sl), _p(kv_cache), kv_cache.shape[0], T, int(compress_ratio),
        int(bool(hadamard))))


def q_rope_fp8_weights(q, w, positions, cos_cache, sin_cache, rope_style,
                       hadamard: bool = False):
    """FP8 mode: (q_out [T,H,128] u8, weights [T,H] f32 with the scale folded in,
    status)."""
    q = _c(q, np.uint16)
    T, H, D = q.shape
    assert D == HEAD_DIM
    w = _c(w, np.uint16)
    pos = _c(positions, np.int64)
    cs = _c(cos_cache, np.float32)
    sn = _c(sin_cache, np.float32)
    qo = np.zeros((T, H, HEAD_DIM), np.uint8)
    wt = np.zeros((T, H), np.float32)
    st = lib().oracle_q_rope_fp8_weights(
        _p(q), _p(w), _p(pos), _p(cs), _p(sn), cs.shape[0], int(rope_style), _p(qo), _p(wt),
        T, H, int(bool(hadamard)))
    return qo, wt, int(st)


def fake_quant_row(row_bits, mode: int) -> np.ndarray:
    """Dequantised bf16 row: mode 0 per-32 UE8M0, mode 1 per-16 E4M3."""
    r = _c(row_bits, np.uint16)
    assert r.shape == (HEAD_DIM,)
    out = np.zeros(HEAD_DIM, np.uint16)
    lib().oracle_fake_quant_row(_p(r), int(mode), _p(out))
    return out


def rope_fake_quant(x, rows_per_token: int, positions, cos_cache, sin_cache, rope_style,
                    mode: int, out=None):
    """(out bf16 bits [N,128], status) for rows x [N,128]."""
    x = _c(x, np.uint16)
    N = x.shape[0]
    assert x.shape == (N, HEAD_DIM)
    pos = _c(positions, np.int64)
    cs = _c(cos_cache, np.float32)
    sn = _c(sin_cache, np.float32)
    if out is None:
        out = np.zeros((N, HEAD_DIM), np.uint16)
    st = lib().oracle_rope_fake_quant(_p(x), int(rows_per_token), _p(pos), _p(cs), _p(sn),
                                      cs.shape[0], int(rope_style), int(mode), _p(out), N)
    return out, int(st)


def paged_mqa_logits(q_fp4, q_scale, weights, kv_cache, block_table, context_lens,
                     next_n: int, max_context: int):
    """Returns (logits fp32 [B*next_n, max_context], status)."""
    qf = _c(q_fp4, np.uint8)
    qs = _c(q_scale, np.uint8)
    wt = _c(weights, np.float32)
    R, H, _ = qf.shape
    assert qf.shape[2] == PAYLOAD_BYTES and qs.shape == (R, H, EXP_BYTES) and wt.shape == (R, H)
    cache = _c(kv_cache, np.uint8)
    assert cache.shape[1:] == (PAGE_BYTES,)
    bt = _c(block_table, np.int32)
    cl = _c(context_lens, np.int32)
    B = cl.shape[0]
    assert R == B * next_n and bt.shape[0] == B
    out = np.empty((R, max_context), np.float32)
    st = lib().oracle_paged_mqa_logits(
        _p(qf), _p(qs), _p(wt), _p(cache), cache.shape[0], _p(bt), bt.shape[1], _p(cl),
        _p(out), max_context, B, next_n, H, max_context)
    return out, int(st)


def mqa_logits_prefill(q_fp4, q_scale, weights, kv_cache, ks, ke, num_keys: int):
    """Prefill scorer: (logits fp32 [T, num_keys], status) for query tokens
    q_fp4 [T,H,64] against the consecutive keys 0..num_keys-1 of kv_cache
    (key s at page s/64, offset s%64), token t scoring [ks[t], ke[t])."""
    qf = _c(q_fp4, np.uint8)
    qs = _c(q_scale, np.uint8)
    wt = _c(weights, np.float32)
    T, H, _ = qf.shape
    assert qf.shape[2] == PAYLOAD_BYTES and qs.shape == (T, H, EXP_BYTES) and wt.shape == (T, H)
    cache = _c(kv_cache, np.uint8)
    assert cache.shape[1:] == (PAGE_BYTES,) and cache.shape[0] * KV_BLOCK >= num_keys
    a = _c(ks, np.int32)
    b = _c(ke, np.int32)
    assert a.shape == (T,) and b.shape == (T,)
    out = np.empty((T, num_keys), np.float32)
    st = lib().oracle_mqa_logits_prefill(_p(qf), _p(qs), _p(wt), _p(cache), int(num_keys),
                                         _p(a), _p(b), _p(out), num_keys, T, H)
    return out, int(st)

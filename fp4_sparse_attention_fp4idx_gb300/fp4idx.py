"""ctypes binding of libfp4idx.so (argument marshalling only).

Importing this module loads the CUDA library and raises ImportError if it is
missing: there is no CPU path.  Build it with
``python -m fp4_sparse_attention_fp4idx_gb300.build``.

Two layers:
  * ``lib()`` -- the raw C ABI (names and argument order of include/fp4idx.h,
    plain integers for pointers).
  * torch wrappers with the same names (minus the ``fp4idx_`` prefix) that
    check dtypes/devices, allocate outputs with torch, pass ``data_ptr()``s
    and the current CUDA stream, and raise ``Fp4idxError`` on a non-OK
    status.  Every step of the computation runs in the library's kernels.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfp4idx.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "fp4idx.h")

ROPE_NEOX = 0
ROPE_INTERLEAVED = 1
HEAD_DIM = 128
PAGE_BYTES = 4352
ERRFLAG_POSITION = 0x1
ERRFLAG_SLOT = 0x2
ERRFLAG_TIMEOUT = 0x4
ERRFLAG_PAGE = 0x8

OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_ARG, ERR_CUDA, ERR_SCRATCH = range(7)
STATIC_STAGING_BYTES = 64 << 20  # FP4IDX_STATIC_STAGING_BYTES

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with "
        "`python -m fp4_sparse_attention_fp4idx_gb300.build` (needs nvcc); "
        "there is no CPU fallback")

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_F = ctypes.c_float
_INT = ctypes.c_int

_SIGS = {
    "fp4idx_k_norm_rope_pack_store": (
        _INT, [_P, _I64, _P, _F, _P, _P, _P, _I64, _INT, _P, _P, _I64, _I64, _P, _P]),
    "fp4idx_q_rope_pack_weights": (
        _INT, [_P, _I64, _I64, _P, _I64, _F, _P, _P, _P, _I64, _INT, _P, _P, _P, _I64,
               _I64, _P, _P]),
    "fp4idx_indexer_prepass": (
        _INT, [_P, _I64, _P, _F, _P, _P, _I64,
               _P, _I64, _I64, _P, _I64, _F, _P, _P, _P, _I64,
               _P, _P, _P, _I64, _INT, _I64, _P, _P]),
    "fp4idx_k_norm_rope_pack_store_ex": (
        _INT, [_P, _I64, _P, _F, _P, _P, _P, _I64, _INT, _P, _P, _I64, _I64, _P, _P, _P]),
    "fp4idx_q_rope_pack_weights_ex": (
        _INT, [_P, _I64, _I64, _P, _I64, _F, _P, _P, _P, _I64, _INT, _P, _P, _P, _I64,
               _I64, _P, _P, _P]),
    "fp4idx_indexer_prepass_ex": (
        _INT, [_P, _I64, _P, _F, _P, _P, _I64,
               _P, _I64, _I64, _P, _I64, _F, _P, _P, _P, _I64,
               _P, _P, _P, _I64, _INT, _I64, _P, _P, _P]),
    "fp4idx_rope_fake_quant": (
        _INT, [_P, _I64, _I64, _P, _P, _P, _I64, _INT, _INT, _P, _I64, _P, _P]),
    "fp4idx_paged_mqa_logits": (
        _INT, [_P, _P, _P, _P, _I64, _P, _I64, _P, _P, _I64, _I64, _I64, _I64, _I64, _P, _P]),
    "fp4idx_mqa_logits_prefill": (
        _INT, [_P, _P, _P, _P, _I64, _I64, _P, _P, _P, _I64, _I64, _I64, _P, _P]),
    "fp4idx_indexer_prepass_host": (
        _INT, [_P, _P, _P, _F, _P, _I64, _P, _P, _I64, _F, _P, _P, _P, _P, _P, _P, _I64,
               _INT, _I64, _I64, _P, _P, _P]),
    "fp4idx_host_staging_bytes": (ctypes.c_size_t, [_I64, _I64]),
    "fp4idx_indexer_prepass_host_static": (
        _INT, [_P, _P, _P, _F, _P, _I64, _P, _P, _I64, _F, _P, _P, _P, _P, _P, _P, _I64,
               _INT, _I64, _I64, _P, _P]),
    "fp4idx_default_weight_scale": (_F, [_I64]),
    "fp4idx_test_withhold_next": (_INT, [_INT, _I64]),
    "fp4idx_status_string": (ctypes.c_char_p, [_INT]),
    "fp4idx_version": (ctypes.c_char_p, []),
}

_lib = ctypes.CDLL(LIB_PATH)
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


def lib() -> ctypes.CDLL:
    return _lib


OUTPUT_FP4 = 0
OUTPUT_FP8 = 1
FP8_PAGE_BYTES = 8448


class Options(ctypes.Structure):
    """fp4idx_options of include/fp4idx.h."""
    _fields_ = [("compress_ratio", ctypes.c_int32), ("hadamard", ctypes.c_int32),
                ("output_mode", ctypes.c_int32)]


def _options(compress_ratio: int, hadamard: bool, fp8: bool = False):
    """None for the defaults (the plain entry points are called), else a
    pointer to an Options block for the _ex entry points."""
    if compress_ratio == 1 and not hadamard and not fp8:
        return None
    return ctypes.pointer(Options(int(compress_ratio), 1 if hadamard else 0,
                                  OUTPUT_FP8 if fp8 else OUTPUT_FP4))


def declared_symbols(header: str = HEADER_PATH) -> list:
    """Names of the functions include/fp4idx.h declares."""
    with open(header) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    return sorted(set(re.findall(r"\b(fp4idx_[a-z0-9_]+)\s*\(", text)))


def status_string(status: int) -> str:
    return _lib.fp4idx_status_string(int(status)).decode()


def version() -> str:
    return _lib.fp4idx_version().decode()


class Fp4idxError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: status {status} ({status_string(status)})")
        self.status = status


def _check(status: int, where: str) -> None:
    if status != OK:
        raise Fp4idxError(status, where)


def rope_style_code(style) -> int:
    if style in (ROPE_NEOX, "neox"):
        return ROPE_NEOX
    if style in (ROPE_INTERLEAVED, "interleaved", "gptj"):
        return ROPE_INTERLEAVED
    raise ValueError(f"unknown rope style {style!r}")


TEST_PREPASS = 0
TEST_SCORER = 1


def test_withhold_next(kernel: int, index: int) -> None:
    """Testing hook: the next launch of `kernel` (TEST_PREPASS: the streaming
    pre-pass; TEST_SCORER: the scorers) leaves out the copies of work item
    `index` of its first CTA, so its bounded waits run out (TIMEOUT flag)."""
    _check(_lib.fp4idx_test_withhold_next(int(kernel), int(index)), "fp4idx_test_withhold_next")


def default_weight_scale(num_heads: int) -> float:
    """The library's head-weight scale, fp32(H^-1/2 * 128^-1/2)."""
    return float(_lib.fp4idx_default_weight_scale(int(num_heads)))


# ------------------------------------------------------------ torch wrappers
def _torch():
    import torch
    return torch


def _stream_ptr(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(int(s.cuda_stream))


def _need(t, dtype, name, ndim=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    return t


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def k_norm_rope_pack_store(k, gamma, positions, cos_cache, sin_cache, slot_mapping,
                           kv_cache, *, eps: float = 1e-6, rope_style="neox",
                           compress_ratio: int = 1, hadamard: bool = False,
                           err_flags=None, stream=None) -> None:
    """Keys -> paged FP4 index cache, in place.  k bf16 [T,128] (row stride a
    multiple of 8), gamma bf16 [128], positions/slot_mapping int64 [T],
    cos/sin fp32 [max_pos,32], kv_cache uint8 [num_blocks, 4352].
    compress_ratio / hadamard select the stated variants (fp4idx_options)."""
    torch = _torch()
    _need(k, torch.bfloat16, "k", 2)
    _need(gamma, torch.bfloat16, "gamma", 1)
    _need(positions, torch.int64, "positions", 1)
    _need(slot_mapping, torch.int64, "slot_mapping", 1)
    _need(cos_cache, torch.float32, "cos_cache", 2)
    _need(sin_cache, torch.float32, "sin_cache", 2)
    _need(kv_cache, torch.uint8, "kv_cache", 2)
    T = k.shape[0]
    if k.shape[1] != HEAD_DIM or k.stride(1) != 1:
        raise ValueError("k must be [T,128] with unit element stride")
    if gamma.shape[0] != HEAD_DIM or not gamma.is_contiguous():
        raise ValueError("gamma must be contiguous [128]")
    if positions.shape[0] != T or slot_mapping.shape[0] != T:
        raise ValueError("positions and slot_mapping must have T entries")
    if not (positions.is_contiguous() and slot_mapping.is_contiguous()):
        raise ValueError("positions and slot_mapping must be contiguous")
    if cos_cache.shape != sin_cache.shape or cos_cache.shape[1] != 32:
        raise ValueError("cos/sin caches must both be [max_pos, 32]")
    if not (cos_cache.is_contiguous() and sin_cache.is_contiguous()):
        raise ValueError("cos/sin caches must be contiguous")
    if kv_cache.shape[1] != PAGE_BYTES or not kv_cache.is_contiguous():
        raise ValueError("kv_cache must be contiguous [num_blocks, 4352]")
    args = (_ptr(k), k.stride(0), _ptr(gamma), float(eps), _ptr(positions), _ptr(cos_cache),
            _ptr(sin_cache), cos_cache.shape[0], rope_style_code(rope_style),
            _ptr(slot_mapping), _ptr(kv_cache), kv_cache.shape[0], T)
    opts = _options(compress_ratio, hadamard)
    if opts is None:
        st = _lib.fp4idx_k_norm_rope_pack_store(*args, _ptr(err_flags), _stream_ptr(stream))
    else:
        st = _lib.fp4idx_k_norm_rope_pack_store_ex(*args, ctypes.cast(opts, _P),
                                                   _ptr(err_flags), _stream_ptr(stream))
    _check(st, "fp4idx_k_norm_rope_pack_store")


def _q_outputs(q_fp4, q_scale, weights, T, H, device):
    torch = _torch()
    if q_fp4 is None:
        q_fp4 = torch.empty((T, H, 64), dtype=torch.uint8, device=device)
    if q_scale is None:
        q_scale = torch.empty((T, H, 4), dtype=torch.uint8, device=device)
    if weights is None:
        weights = torch.empty((T, H), dtype=torch.float32, device=device)
    for t, shape, dt, name in ((q_fp4, (T, H, 64), torch.uint8, "q_fp4"),
                               (q_scale, (T, H, 4), torch.uint8, "q_scale"),
                               (weights, (T, H), torch.float32, "weights")):
        _need(t, dt, name)
        if tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous {shape}")
    return q_fp4, q_scale, weights


def _check_q(q, w, positions, cos_cache, sin_cache):
    torch = _torch()
    _need(q, torch.bfloat16, "q", 3)
    _need(w, torch.bfloat16, "w", 2)
    _need(positions, torch.int64, "positions", 1)
    _need(cos_cache, torch.float32, "cos_cache", 2)
    _need(sin_cache, torch.float32, "sin_cache", 2)
    T, H, D = q.shape
    if D != HEAD_DIM or q.stride(2) != 1:
        raise ValueError("q must be [T,H,128] with unit element stride")
    if tuple(w.shape) != (T, H) or w.stride(1) != 1:
        raise ValueError("w must be [T,H] with unit head stride")
    if positions.shape[0] != T or not positions.is_contiguous():
        raise ValueError("positions must be contiguous [T]")
    if cos_cache.shape != sin_cache.shape or cos_cache.shape[1] != 32:
        raise ValueError("cos/sin caches must both be [max_pos, 32]")
    if not (cos_cache.is_contiguous() and sin_cache.is_contiguous()):
        raise ValueError("cos/sin caches must be contiguous")
    return T, H


def q_rope_pack_weights(q, w, positions, cos_cache, sin_cache, *, rope_style="neox",
                        weight_scale=None, q_fp4=None, q_scale=None, weights=None,
                        hadamard: bool = False, err_flags=None, stream=None):
    """Queries -> (q_fp4 uint8 [T,H,64], q_scale uint8 [T,H,4], weights fp32
    [T,H]).  q bf16 [T,H,128] (strides multiples of 8), w bf16 [T,H]."""
    T, H = _check_q(q, w, positions, cos_cache, sin_cache)
    q_fp4, q_scale, weights = _q_outputs(q_fp4, q_scale, weights, T, H, q.device)
    ws = default_weight_scale(H) if weight_scale is None else float(weight_scale)
    args = (_ptr(q), q.stride(0), q.stride(1), _ptr(w), w.stride(0), ws, _ptr(positions),
            _ptr(cos_cache), _ptr(sin_cache), cos_cache.shape[0], rope_style_code(rope_style),
            _ptr(q_fp4), _ptr(q_scale), _ptr(weights), T, H)
    opts = _options(1, hadamard)
    if opts is None:
        st = _lib.fp4idx_q_rope_pack_weights(*args, _ptr(err_flags), _stream_ptr(stream))
    else:
        st = _lib.fp4idx_q_rope_pack_weights_ex(*args, ctypes.cast(opts, _P), _ptr(err_flags),
                                                _stream_ptr(stream))
    _check(st, "fp4idx_q_rope_pack_weights")
    return q_fp4, q_scale, weights


def indexer_prepass(k, gamma, slot_mapping, kv_cache, q, w, positions, cos_cache, sin_cache, *,
                    eps: float = 1e-6, rope_style="neox", weight_scale=None, q_fp4=None,
                    q_scale=None, weights=None, compress_ratio: int = 1,
                    hadamard: bool = False, err_flags=None, stream=None):
    """Both halves in one launch; returns (q_fp4, q_scale, weights) and updates
    kv_cache in place.  Same argument rules as the two separate calls."""
    torch = _torch()
    T, H = _check_q(q, w, positions, cos_cache, sin_cache)
    _need(k, torch.bfloat16, "k", 2)
    _need(gamma, torch.bfloat16, "gamma", 1)
    _need(slot_mapping, torch.int64, "slot_mapping", 1)
    _need(kv_cache, torch.uint8, "kv_cache", 2)
    if k.shape[0] != T or k.shape[1] != HEAD_DIM or k.stride(1) != 1:
        raise ValueError("k must be [T,128] with unit element stride")
    if gamma.shape[0] != HEAD_DIM or not gamma.is_contiguous():
        raise ValueError("gamma must be contiguous [128]")
    if slot_mapping.shape[0] != T or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be contiguous [T]")
    if kv_cache.shape[1] != PAGE_BYTES or not kv_cache.is_contiguous():
        raise ValueError("kv_cache must be contiguous [num_blocks, 4352]")
    q_fp4, q_scale, weights = _q_outputs(q_fp4, q_scale, weights, T, H, q.device)
    ws = default_weight_scale(H) if weight_scale is None else float(weight_scale)
    args = (_ptr(k), k.stride(0), _ptr(gamma), float(eps), _ptr(slot_mapping), _ptr(kv_cache),
            kv_cache.shape[0], _ptr(q), q.stride(0), q.stride(1), _ptr(w), w.stride(0), ws,
            _ptr(q_fp4), _ptr(q_scale), _ptr(weights), H, _ptr(positions), _ptr(cos_cache),
            _ptr(sin_cache), cos_cache.shape[0], rope_style_code(rope_style), T)
    opts = _options(compress_ratio, hadamard)
    if opts is None:
        st = _lib.fp4idx_indexer_prepass(*args, _ptr(err_flags), _stream_ptr(stream))
    else:
        st = _lib.fp4idx_indexer_prepass_ex(*args, ctypes.cast(opts, _P), _ptr(err_flags),
                                            _stream_ptr(stream))
    _check(st, "fp4idx_indexer_prepass")
    return q_fp4, q_scale, weights


# ------------------------------------------------------- host-buffer pipeline
_STAGING = {}  # (device index, chunk_tokens, H) -> device staging tensor
_STAGING_LOCK = threading.Lock()


def _need_host(t, dtype, name, ndim):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-D tensor")
    return t


def _staging(device, chunk: int, H: int):
    """The device staging buffer of fp4idx_indexer_prepass_host, allocated
    once per (device, chunk, H) and kept (its contents are scratch)."""
    torch = _torch()
    nbytes = int(_lib.fp4idx_host_staging_bytes(chunk, H))
    if nbytes == 0:
        raise ValueError(f"chunk_tokens {chunk} x num_heads {H} is too large")
    key = (device.index, chunk, H)
    with _STAGING_LOCK:
        buf = _STAGING.get(key)
        if buf is None:
            buf = _STAGING[key] = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return buf


def _host_args(k, gamma, slot_mapping, kv_cache, q, w, positions, cos_cache, sin_cache,
               weight_scale, q_fp4, q_scale, weights, chunk_tokens):
    """Checks of the host-buffer calls; returns (T, H, chunk, q_fp4, q_scale,
    weights, weight_scale) with the host outputs allocated pinned when not
    given."""
    torch = _torch()
    _need_host(k, torch.bfloat16, "k", 2)
    _need_host(q, torch.bfloat16, "q", 3)
    _need_host(w, torch.bfloat16, "w", 2)
    _need_host(positions, torch.int64, "positions", 1)
    _need_host(slot_mapping, torch.int64, "slot_mapping", 1)
    _need(kv_cache, torch.uint8, "kv_cache", 2)
    _need(gamma, torch.bfloat16, "gamma", 1)
    T, H, D = q.shape
    if D != HEAD_DIM or tuple(k.shape) != (T, HEAD_DIM) or tuple(w.shape) != (T, H):
        raise ValueError("k must be [T,128], q [T,H,128], w [T,H]")
    if positions.shape[0] != T or slot_mapping.shape[0] != T:
        raise ValueError("positions and slot_mapping must have T entries")
    if gamma.shape[0] != HEAD_DIM or not gamma.is_contiguous():
        raise ValueError("gamma must be contiguous [128]")
    if kv_cache.shape[1] != PAGE_BYTES or not kv_cache.is_contiguous():
        raise ValueError("kv_cache must be contiguous [num_blocks, 4352]")
    for t, name in ((cos_cache, "cos_cache"), (sin_cache, "sin_cache")):
        _need(t, torch.float32, name, 2)
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if chunk_tokens < 1:
        raise ValueError("chunk_tokens must be >= 1")
    outs = []
    for t, shape, dt, name in ((q_fp4, (T, H, 64), torch.uint8, "q_fp4"),
                               (q_scale, (T, H, 4), torch.uint8, "q_scale"),
                               (weights, (T, H), torch.float32, "weights")):
        if t is None:
            t = torch.empty(shape, dtype=dt).pin_memory()
        _need_host(t, dt, name, len(shape))
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} must be {shape}")
        outs.append(t)
    ws = default_weight_scale(H) if weight_scale is None else float(weight_scale)
    return T, H, min(int(chunk_tokens), max(T, 1)), outs[0], outs[1], outs[2], ws


def indexer_prepass_host(k, gamma, slot_mapping, kv_cache, q, w, positions, cos_cache,
                         sin_cache, *, eps: float = 1e-6, rope_style="neox", weight_scale=None,
                         q_fp4=None, q_scale=None, weights=None, chunk_tokens: int = 4096,
                         err_flags=None, stream=None):
    """indexer_prepass for inputs and outputs in host memory, through the
    C-ABI call fp4idx_indexer_prepass_host: k [T,128], q [T,H,128], w [T,H]
    (bf16), positions and slot_mapping [T] (int64) are contiguous host
    tensors, pinned for the copies to overlap; gamma, the cos/sin caches and
    kv_cache are device tensors.  The library pipelines the tokens in chunks
    of chunk_tokens (upload of chunk c+1, fused launch of chunk c, download of
    chunk c-1) on its own streams.  Returns host tensors (q_fp4, q_scale,
    weights), allocated pinned when not given; they are complete once the
    caller's stream (which waits for the pipeline) has reached this point."""
    torch = _torch()
    T, H, chunk, q_fp4, q_scale, weights, ws = _host_args(
        k, gamma, slot_mapping, kv_cache, q, w, positions, cos_cache, sin_cache, weight_scale,
        q_fp4, q_scale, weights, chunk_tokens)
    if T == 0:
        return q_fp4, q_scale, weights
    dev = kv_cache.device
    staging = _staging(dev, chunk, H)
    caller = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        st = _lib.fp4idx_indexer_prepass_host(
            _ptr(k), _ptr(slot_mapping), _ptr(gamma), float(eps), _ptr(kv_cache),
            kv_cache.shape[0], _ptr(q), _ptr(w), H, ws, _ptr(q_fp4), _ptr(q_scale),
            _ptr(weights), _ptr(positions), _ptr(cos_cache), _ptr(sin_cache),
            cos_cache.shape[0], rope_style_code(rope_style), T, chunk, _ptr(staging),
            _ptr(err_flags), _stream_ptr(caller))
    _check(st, "fp4idx_indexer_prepass_host")
    return q_fp4, q_scale, weights


def indexer_prepass_host_static(k, gamma, slot_mapping, kv_cache, q, w, positions, cos_cache,
                                sin_cache, *, eps: float = 1e-6, rope_style="neox",
                                weight_scale=None, q_fp4=None, q_scale=None, weights=None,
                                chunk_tokens=None, err_flags=None, stream=None):
    """indexer_prepass_host with the staging in the library's static device
    buffer (fp4idx_indexer_prepass_host_static): nothing is allocated on the
    device; chunk_tokens must keep the staging within STATIC_STAGING_BYTES
    (ERR_SCRATCH otherwise).  By default it is the largest power-of-two
    share of 1024 tokens whose staging fits."""
    torch = _torch()
    if chunk_tokens is None:
        H = q.shape[1] if hasattr(q, "shape") and q.dim() == 3 else 1
        chunk_tokens = 1024
        while chunk_tokens > 1 and (
                _lib.fp4idx_host_staging_bytes(chunk_tokens, H) == 0 or
                _lib.fp4idx_host_staging_bytes(chunk_tokens, H) > STATIC_STAGING_BYTES):
            chunk_tokens //= 2
    T, H, chunk, q_fp4, q_scale, weights, ws = _host_args(
        k, gamma, slot_mapping, kv_cache, q, w, positions, cos_cache, sin_cache, weight_scale,
        q_fp4, q_scale, weights, chunk_tokens)
    if T == 0:
        return q_fp4, q_scale, weights
    dev = kv_cache.device
    caller = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        st = _lib.fp4idx_indexer_prepass_host_static(
            _ptr(k), _ptr(slot_mapping), _ptr(gamma), float(eps), _ptr(kv_cache),
            kv_cache.shape[0], _ptr(q), _ptr(w), H, ws, _ptr(q_fp4), _ptr(q_scale),
            _ptr(weights), _ptr(positions), _ptr(cos_cache), _ptr(sin_cache),
            cos_cache.shape[0], rope_style_code(rope_style), T, chunk, _ptr(err_flags),
            _stream_ptr(caller))
    _check(st, "fp4idx_indexer_prepass_host_static")
    return q_fp4, q_scale, weights


def paged_mqa_logits(q_fp4, q_scale, weights, kv_cache, block_table, context_lens,
                     max_context: int, *, next_n: int = 1, logits=None, err_flags=None,
                     stream=None):
    """FP4 paged MQA logits -> fp32 [batch*next_n, max_context].  q_fp4 uint8
    [batch*next_n, H, 64], q_scale uint8 [batch*next_n, H, 4], weights fp32
    [batch*next_n, H] (the pre-pass's query outputs), kv_cache uint8
    [num_blocks, 4352], block_table int32 [batch, >= ceil(max_context/64)]
    (unit column stride), context_lens int32 [batch]."""
    torch = _torch()
    _need(q_fp4, torch.uint8, "q_fp4", 3)
    _need(q_scale, torch.uint8, "q_scale", 3)
    _need(weights, torch.float32, "weights", 2)
    _need(kv_cache, torch.uint8, "kv_cache", 2)
    _need(block_table, torch.int32, "block_table", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    T, H, nb = q_fp4.shape
    if nb != 64 or not q_fp4.is_contiguous():
        raise ValueError("q_fp4 must be contiguous [batch*next_n, H, 64]")
    if tuple(q_scale.shape) != (T, H, 4) or not q_scale.is_contiguous():
        raise ValueError("q_scale must be contiguous [batch*next_n, H, 4]")
    if tuple(weights.shape) != (T, H) or not weights.is_contiguous():
        raise ValueError("weights must be contiguous [batch*next_n, H]")
    if next_n < 1 or T % next_n:
        raise ValueError("the query rows must be batch*next_n")
    batch = T // next_n
    if block_table.shape[0] != batch or block_table.stride(1) != 1:
        raise ValueError("block_table must be [batch, pages] with unit column stride")
    if context_lens.shape[0] != batch or not context_lens.is_contiguous():
        raise ValueError("context_lens must be contiguous [batch]")
    if kv_cache.shape[1] != PAGE_BYTES or not kv_cache.is_contiguous():
        raise ValueError("kv_cache must be contiguous [num_blocks, 4352]")
    if logits is None:
        logits = torch.empty((T, max_context), dtype=torch.float32, device=q_fp4.device)
    _need(logits, torch.float32, "logits", 2)
    if logits.shape[0] != T or logits.shape[1] < max_context or logits.stride(1) != 1:
        raise ValueError("logits must be [batch*next_n, >= max_context] with unit column stride")
    # A size-1 leading dimension may carry any stride (numpy gives 0 to a
    # new axis); the row width is the stride the C ABI's checks expect then.
    bt_stride = block_table.stride(0) if batch > 1 else block_table.shape[1]
    out_stride = logits.stride(0) if T > 1 else logits.shape[1]
    st = _lib.fp4idx_paged_mqa_logits(
        _ptr(q_fp4), _ptr(q_scale), _ptr(weights), _ptr(kv_cache), kv_cache.shape[0],
        _ptr(block_table), bt_stride, _ptr(context_lens), _ptr(logits), out_stride, batch,
        next_n, H, int(max_context), _ptr(err_flags), _stream_ptr(stream))
    _check(st, "fp4idx_paged_mqa_logits")
    return logits


def mqa_logits_prefill(q_fp4, q_scale, weights, kv_cache, ks, ke, num_keys: int, *,
                       logits=None, err_flags=None, stream=None):
    """FP4 prefill MQA logits -> fp32 [T, num_keys]: query token t (q_fp4
    uint8 [T, H, 64], q_scale uint8 [T, H, 4], weights fp32 [T, H]) against
    the consecutive keys 0 .. num_keys-1 of kv_cache uint8 [num_blocks, 4352]
    (key s at page s/64, offset s%64), over the keys in [ks[t], ke[t])
    (int32 [T]); -inf elsewhere."""
    torch = _torch()
    _need(q_fp4, torch.uint8, "q_fp4", 3)
    _need(q_scale, torch.uint8, "q_scale", 3)
    _need(weights, torch.float32, "weights", 2)
    _need(kv_cache, torch.uint8, "kv_cache", 2)
    _need(ks, torch.int32, "ks", 1)
    _need(ke, torch.int32, "ke", 1)
    T, H, nb = q_fp4.shape
    if nb != 64 or not q_fp4.is_contiguous():
        raise ValueError("q_fp4 must be contiguous [T, H, 64]")
    if tuple(q_scale.shape) != (T, H, 4) or not q_scale.is_contiguous():
        raise ValueError("q_scale must be contiguous [T, H, 4]")
    if tuple(weights.shape) != (T, H) or not weights.is_contiguous():
        raise ValueError("weights must be contiguous [T, H]")
    if tuple(ks.shape) != (T,) or tuple(ke.shape) != (T,) or not (
            ks.is_contiguous() and ke.is_contiguous()):
        raise ValueError("ks and ke must be contiguous [T]")
    if kv_cache.shape[1] != PAGE_BYTES or not kv_cache.is_contiguous():
        raise ValueError("kv_cache must be contiguous [num_blocks, 4352]")
    if logits is None:
        logits = torch.empty((T, num_keys), dtype=torch.float32, device=q_fp4.device)
    _need(logits, torch.float32, "logits", 2)
    if logits.shape[0] != T or logits.shape[1] < num_keys or logits.stride(1) != 1:
        raise ValueError("logits must be [T, >= num_keys] with unit column stride")
    out_stride = logits.stride(0) if T > 1 else logits.shape[1]
    st = _lib.fp4idx_mqa_logits_prefill(
        _ptr(q_fp4), _ptr(q_scale), _ptr(weights), _ptr(kv_cache), kv_cache.shape[0],
        int(num_keys), _ptr(ks), _ptr(ke), _ptr(logits), out_stride, T, H, _ptr(err_flags),
        _stream_ptr(stream))
    _check(st, "fp4idx_mqa_logits_prefill")
    return logits


# ------------------------------------------------------------ FP8 output mode
def k_norm_rope_fp8_store(k, gamma, positions, cos_cache, sin_cache, slot_mapping, kv_cache, *,
                          eps: float = 1e-6, rope_style="neox", compress_ratio: int = 1,
                          hadamard: bool = False, err_flags=None, stream=None) -> None:
    """Keys -> FP8 paged index cache (uint8 [num_blocks, 8448]), in place:
    fp4idx_k_norm_rope_pack_store_ex with output_mode FP8."""
    torch = _torch()
    _need(k, torch.bfloat16, "k", 2)
    _need(kv_cache, torch.uint8, "kv_cache", 2)
    if kv_cache.shape[1] != FP8_PAGE_BYTES or not kv_cache.is_contiguous():
        raise ValueError("kv_cache must be contiguous [num_blocks, 8448]")
    T = k.shape[0]
    if k.shape[1] != HEAD_DIM or k.stride(1) != 1:
        raise ValueError("k must be [T,128] with unit element stride")
    opts = _options(compress_ratio, hadamard, fp8=True)
    st = _lib.fp4idx_k_norm_rope_pack_store_ex(
        _ptr(k), k.stride(0), _ptr(gamma), float(eps), _ptr(positions), _ptr(cos_cache),
        _ptr(sin_cache), cos_cache.shape[0], rope_style_code(rope_style), _ptr(slot_mapping),
        _ptr(kv_cache), kv_cache.shape[0], T, ctypes.cast(opts, _P), _ptr(err_flags),
        _stream_ptr(stream))
    _check(st, "fp4idx_k_norm_rope_pack_store_ex (FP8)")


def _fp8_q_outputs(q_out, weights, T, H, device):
    torch = _torch()
    if q_out is None:
        q_out = torch.empty((T, H, HEAD_DIM), dtype=torch.uint8, device=device)
    if weights is None:
        weights = torch.empty((T, H), dtype=torch.float32, device=device)
    for t, shape, dt, name in ((q_out, (T, H, HEAD_DIM), torch.uint8, "q_out"),
                               (weights, (T, H), torch.float32, "weights")):
        _need(t, dt, name)
        if tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous {shape}")
    return q_out, weights


def q_rope_fp8_weights(q, w, positions, cos_cache, sin_cache, *, rope_style="neox",
                       weight_scale=None, q_out=None, weights=None, hadamard: bool = False,
                       err_flags=None, stream=None):
    """Queries -> (E4M3 codes uint8 [T,H,128], weights fp32 [T,H] with each
    row's power-of-two scale folded in)."""
    T, H = _check_q(q, w, positions, cos_cache, sin_cache)
    q_out, weights = _fp8_q_outputs(q_out, weights, T, H, q.device)
    ws = default_weight_scale(H) if weight_scale is None else float(weight_scale)
    opts = _options(1, hadamard, fp8=True)
    st = _lib.fp4idx_q_rope_pack_weights_ex(
        _ptr(q), q.stride(0), q.stride(1), _ptr(w), w.stride(0), ws, _ptr(positions),
        _ptr(cos_cache), _ptr(sin_cache), cos_cache.shape[0], rope_style_code(rope_style),
        _ptr(q_out), None, _ptr(weights), T, H, ctypes.cast(opts, _P), _ptr(err_flags),
        _stream_ptr(stream))
    _check(st, "fp4idx_q_rope_pack_weights_ex (FP8)")
    return q_out, weights


def indexer_prepass_fp8(k, gamma, slot_mapping, kv_cache, q, w, positions, cos_cache,
                        sin_cache, *, eps: float = 1e-6, rope_style="neox", weight_scale=None,
                        q_out=None, weights=None, compress_ratio: int = 1,
                        hadamard: bool = False, err_flags=None, stream=None):
    """Both halves in the FP8 mode, one launch; returns (q_out, weights) and
    updates kv_cache ([num_blocks, 8448]) in place."""
    torch = _torch()
    T, H = _check_q(q, w, positions, cos_cache, sin_cache)
    _need(k, torch.bfloat16, "k", 2)
    _need(kv_cache, torch.uint8, "kv_cache", 2)
    if kv_cache.shape[1] != FP8_PAGE_BYTES or not kv_cache.is_contiguous():
        raise ValueError("kv_cache must be contiguous [num_blocks, 8448]")
    if k.shape[0] != T or k.shape[1] != HEAD_DIM or k.stride(1) != 1:
        raise ValueError("k must be [T,128] with unit element stride")
    q_out, weights = _fp8_q_outputs(q_out, weights, T, H, q.device)
    ws = default_weight_scale(H) if weight_scale is None else float(weight_scale)
    opts = _options(compress_ratio, hadamard, fp8=True)
    st = _lib.fp4idx_indexer_prepass_ex(
        _ptr(k), k.stride(0), _ptr(gamma), float(eps), _ptr(slot_mapping), _ptr(kv_cache),
        kv_cache.shape[0], _ptr(q), q.stride(0), q.stride(1), _ptr(w), w.stride(0), ws,
        _ptr(q_out), None, _ptr(weights), H, _ptr(positions), _ptr(cos_cache), _ptr(sin_cache),
        cos_cache.shape[0], rope_style_code(rope_style), T, ctypes.cast(opts, _P),
        _ptr(err_flags), _stream_ptr(stream))
    _check(st, "fp4idx_indexer_prepass_ex (FP8)")
    return q_out, weights


# ------------------------------------------------------ torch-shaped fake quant
FAKE_QUANT_UE8M0_32 = 0
FAKE_QUANT_E4M3_16 = 1


def rope_fake_quant(x, positions, cos_cache, sin_cache, *, rope_style="neox",
                    scale_mode: int = FAKE_QUANT_UE8M0_32, out=None, err_flags=None,
                    stream=None):
    """RoPE + FP4 fake quantisation -> bf16 of x's shape.  x bf16 [T,128]
    (keys, one position per row) or [T,H,128] (queries, one position per
    token), unit element stride, row stride a multiple of 8."""
    torch = _torch()
    _need(x, torch.bfloat16, "x")
    if x.dim() == 2:
        T, D = x.shape
        rows, per, stride = T, 1, x.stride(0)
    elif x.dim() == 3:
        T, H, D = x.shape
        if x.stride(0) != H * x.stride(1):
            raise ValueError("x [T,H,128] must have token stride H * head stride")
        rows, per, stride = T * H, H, x.stride(1)
    else:
        raise ValueError("x must be [T,128] or [T,H,128]")
    if D != HEAD_DIM or x.stride(-1) != 1:
        raise ValueError("rows must be 128 elements with unit stride")
    _need(positions, torch.int64, "positions", 1)
    if positions.shape[0] != T or not positions.is_contiguous():
        raise ValueError("positions must be contiguous [T]")
    if out is None:
        out = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, "out")
    if tuple(out.shape) != tuple(x.shape) or not out.is_contiguous():
        raise ValueError("out must be contiguous with x's shape")
    st = _lib.fp4idx_rope_fake_quant(
        _ptr(x), stride, per, _ptr(positions), _ptr(cos_cache), _ptr(sin_cache),
        cos_cache.shape[0], rope_style_code(rope_style), int(scale_mode), _ptr(out), rows,
        _ptr(err_flags), _stream_ptr(stream))
    _check(st, "fp4idx_rope_fake_quant")
    return out

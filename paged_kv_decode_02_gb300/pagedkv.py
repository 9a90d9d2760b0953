"""ctypes binding over libpagedkv.so (see include/pagedkv.h for the C ABI).

Argument marshalling only: every step of append and decode runs in the library's CUDA
kernels. PyTorch supplies device memory (outputs and the workspace come from its
caching allocator) and the current CUDA stream. There is no fallback: if the library
is missing or a tensor is not on a CUDA device, the call raises.
"""

from __future__ import annotations

import ctypes
import enum
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.environ.get("PAGEDKV_LIB", os.path.join(_HERE, "libpagedkv.so"))


class Status(enum.IntEnum):
    OK = 0
    ERR_NULL = -1
    ERR_DTYPE = -2
    ERR_SHAPE = -3
    ERR_UNSUPPORTED = -4
    ERR_WORKSPACE = -5
    ERR_CUDA = -6
    ERR_ALIGNMENT = -7
    ERR_HOST_MEMORY = -8


DEV_BAD_CONTEXT_LEN = 0x1
DEV_BAD_BLOCK_ID = 0x2
DEV_TIMEOUT = 0x4
DEV_BAD_PREFIX = 0x8

KV_BF16 = 0
KV_INT8 = 1
KV_FP8_E4M3 = 2
KV_FP8_E5M2 = 3
FP8_FORMATS = {"e4m3": KV_FP8_E4M3, "e5m2": KV_FP8_E5M2}


_KV_OF_DTYPE = {torch.bfloat16: KV_BF16, torch.int8: KV_INT8, torch.uint8: None,
                torch.float8_e4m3fn: KV_FP8_E4M3, torch.float8_e5m2: KV_FP8_E5M2}


class PagedKVError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_lib().pkv_status_string(status).decode()}")


class Dims(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32)]


EXPORTS = {
    "pkv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pkv_version": (ctypes.c_int, []),
    "pkv_kernel_launch_count": (ctypes.c_uint64, []),
    "pkv_append_bf16": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int32, ctypes.c_void_p,
                                                                ctypes.c_void_p]),
    "pkv_append_int8": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_int32, ctypes.c_void_p,
                                                                ctypes.c_void_p]),
    "pkv_decode_workspace_bytes": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int,
                                                  ctypes.POINTER(ctypes.c_size_t)]),
    "pkv_decode_bf16": (ctypes.c_int, [ctypes.c_void_p] * 6 + [ctypes.c_float, ctypes.c_void_p,
                                                                ctypes.c_void_p, ctypes.c_size_t,
                                                                ctypes.c_void_p, ctypes.c_void_p]),
    "pkv_decode_int8": (ctypes.c_int, [ctypes.c_void_p] * 8 + [ctypes.c_float, ctypes.c_void_p,
                                                                ctypes.c_void_p, ctypes.c_size_t,
                                                                ctypes.c_void_p, ctypes.c_void_p]),
    "pkv_append_fp8": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_int32, ctypes.c_int,
                                                               ctypes.c_void_p, ctypes.c_void_p]),
    "pkv_decode_fp8": (ctypes.c_int, [ctypes.c_void_p] * 8 + [ctypes.c_float, ctypes.c_int,
                                                               ctypes.c_void_p, ctypes.c_void_p,
                                                               ctypes.c_size_t, ctypes.c_void_p,
                                                               ctypes.c_void_p]),
    "pkv_copy_blocks": (ctypes.c_int, [ctypes.c_void_p] * 6 + [ctypes.c_int32, ctypes.c_int,
                                                                ctypes.c_void_p, ctypes.c_void_p,
                                                                ctypes.c_void_p]),
    "pkv_swap_out": (ctypes.c_int, [ctypes.c_void_p] * 9 + [ctypes.c_int32, ctypes.c_int,
                                                             ctypes.c_void_p, ctypes.c_void_p,
                                                             ctypes.c_void_p]),
    "pkv_swap_in": (ctypes.c_int, [ctypes.c_void_p] * 9 + [ctypes.c_int32, ctypes.c_int,
                                                            ctypes.c_void_p, ctypes.c_void_p,
                                                            ctypes.c_void_p]),
    "pkv_decode_multi_workspace_bytes": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32,
                                                        ctypes.POINTER(ctypes.c_size_t)]),
    "pkv_decode_multi_bf16": (ctypes.c_int, [ctypes.c_void_p] * 6 + [ctypes.c_int32,
                                                                      ctypes.c_float,
                                                                      ctypes.c_void_p,
                                                                      ctypes.c_void_p,
                                                                      ctypes.c_size_t,
                                                                      ctypes.c_void_p,
                                                                      ctypes.c_void_p]),
    "pkv_decode_multi_q8_workspace_bytes": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32,
                                                           ctypes.c_int,
                                                           ctypes.POINTER(ctypes.c_size_t)]),
    "pkv_decode_multi_q8": (ctypes.c_int, [ctypes.c_void_p] * 8 + [ctypes.c_int32,
                                                                   ctypes.c_float, ctypes.c_int,
                                                                   ctypes.c_void_p,
                                                                   ctypes.c_void_p,
                                                                   ctypes.c_size_t,
                                                                   ctypes.c_void_p,
                                                                   ctypes.c_void_p]),
    "pkv_decode_cascade_q8_workspace_bytes": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32,
                                                             ctypes.c_int,
                                                             ctypes.POINTER(ctypes.c_size_t)]),
    "pkv_decode_cascade_q8": (ctypes.c_int, [ctypes.c_void_p] * 8 + [ctypes.c_int32,
                                                                     ctypes.c_float, ctypes.c_int,
                                                                     ctypes.c_void_p,
                                                                     ctypes.c_void_p,
                                                                     ctypes.c_size_t,
                                                                     ctypes.c_void_p,
                                                                     ctypes.c_void_p]),
    "pkv_decode_cascade_workspace_bytes": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32,
                                                          ctypes.POINTER(ctypes.c_size_t)]),
    "pkv_decode_cascade_bf16": (ctypes.c_int, [ctypes.c_void_p] * 6 + [ctypes.c_int32,
                                                                        ctypes.c_float,
                                                                        ctypes.c_void_p,
                                                                        ctypes.c_void_p,
                                                                        ctypes.c_size_t,
                                                                        ctypes.c_void_p,
                                                                        ctypes.c_void_p]),
    "pkv_decode_bf16_noalloc": (ctypes.c_int, [ctypes.c_void_p] * 6 + [ctypes.c_float,
                                                                        ctypes.c_void_p,
                                                                        ctypes.c_void_p,
                                                                        ctypes.c_void_p]),
}

_LIB = None
_LOCK = threading.Lock()


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libpagedkv.so (raises if it has not been built)."""
    global _LIB
    with _LOCK:
        if _LIB is not None and path is None:
            return _LIB
        p = path or library_path()
        if not os.path.exists(p):
            raise ImportError(f"{p} not found: build it with `python -m "
                              f"paged_kv_decode_02_gb300.build_lib` (there is no CPU fallback)")
        lib = ctypes.CDLL(p)
        for name, (res, args) in EXPORTS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _LIB = lib
        return lib


def _lib():
    return _LIB if _LIB is not None else load_library()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


class _OnDevice:
    """Make `device` current for the library call (a no-op when it already is)."""

    __slots__ = ("dev", "prev")

    def __init__(self, device):
        self.dev = device.index if device.index is not None else torch.cuda.current_device()
        self.prev = None

    def __enter__(self):
        cur = torch.cuda.current_device()
        if cur != self.dev:
            self.prev = cur
            torch.cuda.set_device(self.dev)

    def __exit__(self, *exc):
        if self.prev is not None:
            torch.cuda.set_device(self.prev)
        return False


def _check(status, what):
    if status != 0:
        raise PagedKVError(status, what)


def _require(t, name, dtype, ndim, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device (no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _dims(num_seqs, num_q_heads, k_cache, max_blocks_per_seq):
    nb, hkv, bs, d = k_cache.shape
    return Dims(num_seqs, num_q_heads, hkv, d, bs, nb, max_blocks_per_seq)


def _same_shape(t, name, shape):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _cache_shapes(k_cache, v_cache, k_scale=None, v_scale=None):
    """V cache and scales against the K cache [NB, Hkv, bs, D]: the kernels address all
    of them through the K cache's sizes."""
    _same_shape(v_cache, "v_cache", k_cache.shape)
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        if t is not None:
            _same_shape(t, n, k_cache.shape[:3])


def _append_shapes(k, v, k_cache, v_cache, slot_mapping, k_scale=None, v_scale=None):
    """New rows [T, Hkv, D] and T slots, against the caches."""
    _cache_shapes(k_cache, v_cache, k_scale, v_scale)
    row = (k.shape[0], k_cache.shape[1], k_cache.shape[3])
    _same_shape(k, "k", row)
    _same_shape(v, "v", row)
    _same_shape(slot_mapping, "slot_mapping", (k.shape[0],))


def paged_kv_append(k, v, k_cache, v_cache, slot_mapping):
    """Write new tokens' K/V rows ([T, Hkv, D] bf16) into the bf16 paged caches
    ([NB, Hkv, bs, D]) at ``slot_mapping`` ([T] int64, -1 = skip). In place."""
    dev = k_cache.device
    for t, n, dt, nd in ((k, "k", torch.bfloat16, 3), (v, "v", torch.bfloat16, 3),
                         (k_cache, "k_cache", torch.bfloat16, 4),
                         (v_cache, "v_cache", torch.bfloat16, 4),
                         (slot_mapping, "slot_mapping", torch.int64, 1)):
        _require(t, n, dt, nd, dev)
    _append_shapes(k, v, k_cache, v_cache, slot_mapping)
    dims = _dims(0, k_cache.shape[1], k_cache, 1)
    with _OnDevice(dev):
        st = _lib().pkv_append_bf16(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(slot_mapping), k.shape[0], ctypes.byref(dims),
                                    _stream(dev))
    _check(st, "pkv_append_bf16")


def paged_kv_append_int8(k, v, k_cache, v_cache, k_scale, v_scale, slot_mapping):
    """Quantise new tokens' K/V rows per (token, KV head) and write INT8 codes into
    ``k_cache``/``v_cache`` ([NB, Hkv, bs, D] int8) and fp32 scales into
    ``k_scale``/``v_scale`` ([NB, Hkv, bs]). In place."""
    dev = k_cache.device
    for t, n, dt, nd in ((k, "k", torch.bfloat16, 3), (v, "v", torch.bfloat16, 3),
                         (k_cache, "k_cache", torch.int8, 4), (v_cache, "v_cache", torch.int8, 4),
                         (k_scale, "k_scale", torch.float32, 3),
                         (v_scale, "v_scale", torch.float32, 3),
                         (slot_mapping, "slot_mapping", torch.int64, 1)):
        _require(t, n, dt, nd, dev)
    _append_shapes(k, v, k_cache, v_cache, slot_mapping, k_scale, v_scale)
    dims = _dims(0, k_cache.shape[1], k_cache, 1)
    with _OnDevice(dev):
        st = _lib().pkv_append_int8(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(k_scale), _ptr(v_scale), _ptr(slot_mapping), k.shape[0],
                                    ctypes.byref(dims), _stream(dev))
    _check(st, "pkv_append_int8")


def paged_kv_append_fp8(k, v, k_cache, v_cache, k_scale, v_scale, slot_mapping, fmt="e5m2"):
    """Quantise new tokens' K/V rows per (token, KV head) to FP8 (``fmt`` "e4m3" or
    "e5m2") and write the codes into ``k_cache``/``v_cache`` ([NB, Hkv, bs, D] uint8 or
    the matching torch float8 dtype) and fp32 scales into ``k_scale``/``v_scale``
    ([NB, Hkv, bs]). In place."""
    kv = _fp8_format(fmt)
    dev = k_cache.device
    for t, n, dt, nd in ((k, "k", torch.bfloat16, 3), (v, "v", torch.bfloat16, 3),
                         (k_scale, "k_scale", torch.float32, 3),
                         (v_scale, "v_scale", torch.float32, 3),
                         (slot_mapping, "slot_mapping", torch.int64, 1)):
        _require(t, n, dt, nd, dev)
    _require_any(k_cache, "k_cache", _code_dtypes(kv), 4, dev)
    _require_any(v_cache, "v_cache", _code_dtypes(kv), 4, dev)
    _append_shapes(k, v, k_cache, v_cache, slot_mapping, k_scale, v_scale)
    dims = _dims(0, k_cache.shape[1], k_cache, 1)
    with _OnDevice(dev):
        st = _lib().pkv_append_fp8(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(k_scale), _ptr(v_scale), _ptr(slot_mapping), k.shape[0],
                                   kv, ctypes.byref(dims), _stream(dev))
    _check(st, "pkv_append_fp8")


def decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                           num_blocks, max_blocks_per_seq, kv_dtype=KV_BF16, device=None):
    dims = Dims(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                max_blocks_per_seq)
    out = ctypes.c_size_t(0)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        st = _lib().pkv_decode_workspace_bytes(ctypes.byref(dims), kv_dtype, ctypes.byref(out))
    _check(st, "pkv_decode_workspace_bytes")
    return int(out.value)


def _fp8_format(fmt):
    if fmt not in FP8_FORMATS:
        raise ValueError(f"fp8 format must be one of {sorted(FP8_FORMATS)}, got {fmt!r}")
    return FP8_FORMATS[fmt]


def _code_dtypes(kv):
    """Cache tensor dtypes accepted for a KV dtype code."""
    if kv == KV_BF16:
        return (torch.bfloat16,)
    if kv == KV_INT8:
        return (torch.int8,)
    return (torch.uint8, torch.float8_e4m3fn if kv == KV_FP8_E4M3 else torch.float8_e5m2)


def _require_any(t, name, dtypes, ndim, device):
    if isinstance(t, torch.Tensor) and t.dtype in dtypes[1:]:
        dtypes = (t.dtype,)
    _require(t, name, dtypes[0], ndim, device)


def _status_word(status, device):
    """The optional device status word: None, or an int32 CUDA tensor on ``device``."""
    if status is None:
        return None
    if not isinstance(status, torch.Tensor) or not status.is_cuda or status.device != device:
        raise ValueError(f"status must be an int32 CUDA tensor on {device}")
    if status.dtype != torch.int32 or status.numel() < 1 or not status.is_contiguous():
        raise TypeError("status must be a contiguous int32 tensor of at least one element")
    return status


def _workspace(workspace, need, device):
    """(tensor, size in bytes) of the decode workspace: the caller's, checked to be a
    contiguous CUDA tensor on ``device``, when it holds ``need`` bytes; else a fresh
    uint8 buffer from torch's allocator."""
    if workspace is not None:
        if (not isinstance(workspace, torch.Tensor) or not workspace.is_cuda
                or workspace.device != device):
            raise ValueError(f"workspace must be a CUDA tensor on {device}")
        if not workspace.is_contiguous():
            raise ValueError("workspace must be contiguous")
        nbytes = workspace.numel() * workspace.element_size()
        if nbytes >= need:
            return workspace, nbytes
    ws = torch.empty(max(int(need), 256), dtype=torch.uint8, device=device)
    return ws, ws.numel()


def _decode(kv, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale,
            out, workspace, status):
    dev = q.device
    status = _status_word(status, dev)
    _require(q, "q", torch.bfloat16, 3, dev)
    _require_any(k_cache, "k_cache", _code_dtypes(kv), 4, dev)
    _require_any(v_cache, "v_cache", _code_dtypes(kv), 4, dev)
    if kv != KV_BF16:
        _require(k_scale, "k_scale", torch.float32, 3, dev)
        _require(v_scale, "v_scale", torch.float32, 3, dev)
    _require(block_tables, "block_tables", torch.int32, 2, dev)
    _require(context_lens, "context_lens", torch.int32, 1, dev)
    B, Hq, D = q.shape
    if k_cache.shape != v_cache.shape or k_cache.shape[3] != D:
        raise ValueError("cache shapes disagree with q")
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables / context_lens must have num_seqs rows")
    _cache_shapes(k_cache, v_cache, k_scale if kv != KV_BF16 else None,
                  v_scale if kv != KV_BF16 else None)
    dims = _dims(B, Hq, k_cache, block_tables.shape[1])
    if out is None:
        out = torch.empty_like(q)
    else:
        _require(out, "out", torch.bfloat16, 3, dev)
        _same_shape(out, "out", q.shape)
    with _OnDevice(dev):
        need = ctypes.c_size_t(0)
        _check(_lib().pkv_decode_workspace_bytes(ctypes.byref(dims), kv, ctypes.byref(need)),
               "pkv_decode_workspace_bytes")
        workspace, ws_bytes = _workspace(workspace, need.value, dev)
        if kv == KV_INT8:
            name = "pkv_decode_int8"
            st = _lib().pkv_decode_int8(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(k_scale), _ptr(v_scale), _ptr(block_tables),
                                        _ptr(context_lens), float(scale), ctypes.byref(dims),
                                        _ptr(workspace), ws_bytes, _ptr(status),
                                        _stream(dev))
        elif kv == KV_BF16:
            name = "pkv_decode_bf16"
            st = _lib().pkv_decode_bf16(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(block_tables), _ptr(context_lens), float(scale),
                                        ctypes.byref(dims), _ptr(workspace), ws_bytes,
                                        _ptr(status), _stream(dev))
        else:
            name = "pkv_decode_fp8"
            st = _lib().pkv_decode_fp8(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                       _ptr(k_scale), _ptr(v_scale), _ptr(block_tables),
                                       _ptr(context_lens), float(scale), kv, ctypes.byref(dims),
                                       _ptr(workspace), ws_bytes, _ptr(status),
                                       _stream(dev))
    _check(st, name)
    return out


def paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale, out=None,
                           workspace=None, status=None):
    """Single-token decode attention over a bf16 paged KV cache (MHA and GQA).

    q [B, Hq, D] bf16; caches [NB, Hkv, bs, D] bf16; block_tables [B, MBS] int32;
    context_lens [B] int32. Returns out [B, Hq, D] bf16. ``workspace`` (uint8, at
    least :func:`decode_workspace_bytes`) and
    ``status`` (int32 [1]) are optional.
    """
    return _decode(KV_BF16, q, k_cache, v_cache, None, None, block_tables, context_lens, scale,
                   out, workspace, status)


def paged_decode_attention_int8(q, k_cache, v_cache, k_scale, v_scale, block_tables,
                                context_lens, scale, out=None, workspace=None, status=None):
    """As :func:`paged_decode_attention` over an INT8 cache with per-(token, KV head)
    fp32 scales ``k_scale``/``v_scale`` [NB, Hkv, bs]."""
    return _decode(KV_INT8, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                   scale, out, workspace, status)


def paged_decode_attention_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables,
                               context_lens, scale, fmt="e5m2", out=None, workspace=None,
                               status=None):
    """As :func:`paged_decode_attention` over an FP8 cache (``fmt`` "e4m3" or "e5m2";
    codes as uint8 or the matching torch float8 dtype) with per-(token, KV head) fp32
    scales ``k_scale``/``v_scale`` [NB, Hkv, bs]."""
    return _decode(_fp8_format(fmt), q, k_cache, v_cache, k_scale, v_scale, block_tables,
                   context_lens, scale, out, workspace, status)


def _move_kv(k_cache, kv_dtype):
    """KV dtype code of a block move: from the cache dtype, or ``kv_dtype`` (needed for
    uint8 FP8 codes, where any one-byte code gives the same move)."""
    if not isinstance(k_cache, torch.Tensor):
        raise TypeError("k_cache must be a torch.Tensor")
    kv = _KV_OF_DTYPE.get(k_cache.dtype, -1) if kv_dtype is None else kv_dtype
    if kv is None:
        kv = KV_FP8_E5M2                      # uint8 codes: one byte + scales
    if kv == -1:
        raise TypeError(f"unsupported cache dtype {k_cache.dtype}")
    return kv


def _move_dims(k_cache):
    nb, hkv, bs, d = k_cache.shape
    return Dims(0, hkv, hkv, d, bs, nb, 1)


def _move_caches(kv, k_cache, v_cache, k_scale, v_scale):
    """Checks the device side of a block move; returns (device, bytes of one block of
    one cache, bytes of one block's scales or 0)."""
    dev = k_cache.device
    _require(k_cache, "k_cache", k_cache.dtype, 4, dev)
    _require(v_cache, "v_cache", k_cache.dtype, 4, dev)
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache differ in shape")
    nb, hkv, bs, d = k_cache.shape
    block = hkv * bs * d * k_cache.element_size()
    if kv == KV_BF16:
        return dev, block, 0
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _require(t, n, torch.float32, 3, dev)
        if tuple(t.shape) != (nb, hkv, bs):
            raise ValueError(f"{n} must be [num_blocks, num_kv_heads, block_size]")
    return dev, block, hkv * bs * 4


def _host_buffers(kv, n, block, scale_block, host_k, host_v, host_k_scale, host_v_scale):
    """Checks that the pinned host buffers of a swap hold ``n`` packed blocks (the GPU
    reads or writes them directly, so a short buffer would be overrun)."""
    bufs = [(host_k, "host_k", block), (host_v, "host_v", block)]
    if kv != KV_BF16:
        bufs += [(host_k_scale, "host_k_scale", scale_block),
                 (host_v_scale, "host_v_scale", scale_block)]
    for t, name, per_block in bufs:
        _host(t, name)
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.numel() * t.element_size() < n * per_block:
            raise ValueError(f"{name} holds {t.numel() * t.element_size()} bytes, "
                             f"{n} blocks need {n * per_block}")


def cascade_q8_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                               num_blocks, max_blocks_per_seq, prefix_blocks, kv_dtype,
                               device=None):
    """Workspace of :func:`paged_decode_attention_cascade_q8` (kv_dtype KV_INT8,
    KV_FP8_E4M3 or KV_FP8_E5M2)."""
    dims = Dims(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                max_blocks_per_seq)
    out = ctypes.c_size_t(0)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        st = _lib().pkv_decode_cascade_q8_workspace_bytes(ctypes.byref(dims), int(prefix_blocks),
                                                          int(kv_dtype), ctypes.byref(out))
    _check(st, "pkv_decode_cascade_q8_workspace_bytes")
    return int(out.value)


def paged_decode_attention_cascade_q8(q, k_cache, v_cache, k_scale, v_scale, block_tables,
                                      context_lens, prefix_blocks, scale, fmt="e5m2", out=None,
                                      workspace=None, status=None):
    """:func:`paged_decode_attention_cascade` over a one-byte cache: int8 codes (INT8),
    or FP8 codes (uint8 with ``fmt`` "e4m3" / "e5m2", or the matching torch float8
    dtype), with per-(token, KV head) fp32 scales ``k_scale``/``v_scale`` [NB, Hkv, bs].
    Same result as :func:`paged_decode_attention_int8` / :func:`paged_decode_attention_fp8`."""
    dev = q.device
    status = _status_word(status, dev)
    kv = _q8_kind(k_cache, fmt)
    _require(q, "q", torch.bfloat16, 3, dev)
    _require_any(k_cache, "k_cache", _code_dtypes(kv), 4, dev)
    _require_any(v_cache, "v_cache", _code_dtypes(kv), 4, dev)
    _require(k_scale, "k_scale", torch.float32, 3, dev)
    _require(v_scale, "v_scale", torch.float32, 3, dev)
    _require(block_tables, "block_tables", torch.int32, 2, dev)
    _require(context_lens, "context_lens", torch.int32, 1, dev)
    B, Hq, D = q.shape
    if k_cache.shape != v_cache.shape or k_cache.shape[3] != D:
        raise ValueError("cache shapes disagree with q")
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables / context_lens must have num_seqs rows")
    _cache_shapes(k_cache, v_cache, k_scale, v_scale)
    dims = _dims(B, Hq, k_cache, block_tables.shape[1])
    if out is None:
        out = torch.empty_like(q)
    else:
        _require(out, "out", torch.bfloat16, 3, dev)
        _same_shape(out, "out", q.shape)
    with _OnDevice(dev):
        need = ctypes.c_size_t(0)
        _check(_lib().pkv_decode_cascade_q8_workspace_bytes(ctypes.byref(dims),
                                                            int(prefix_blocks), kv,
                                                            ctypes.byref(need)),
               "pkv_decode_cascade_q8_workspace_bytes")
        workspace, ws_bytes = _workspace(workspace, need.value, dev)
        st = _lib().pkv_decode_cascade_q8(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                          _ptr(k_scale), _ptr(v_scale), _ptr(block_tables),
                                          _ptr(context_lens), int(prefix_blocks), float(scale),
                                          kv, ctypes.byref(dims), _ptr(workspace), ws_bytes,
                                          _ptr(status), _stream(dev))
    _check(st, "pkv_decode_cascade_q8")
    return out


def copy_blocks(k_cache, v_cache, src_ids, dst_ids, k_scale=None, v_scale=None, status=None,
                kv_dtype=None):
    """Copy-on-write block copy: block dst_ids[i] := block src_ids[i] of the K/V caches
    (and their scales, for one-byte caches). ``src_ids``/``dst_ids``: device int32.
    In place, asynchronous on the current stream."""
    kv = _move_kv(k_cache, kv_dtype)
    dev, _, _ = _move_caches(kv, k_cache, v_cache, k_scale, v_scale)
    status = _status_word(status, dev)
    for t, n in ((src_ids, "src_ids"), (dst_ids, "dst_ids")):
        _require(t, n, torch.int32, 1, dev)
    if src_ids.numel() != dst_ids.numel():
        raise ValueError("src_ids and dst_ids differ in length")
    dims = _move_dims(k_cache)
    with _OnDevice(dev):
        st = _lib().pkv_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                    _ptr(src_ids), _ptr(dst_ids), src_ids.numel(), kv,
                                    ctypes.byref(dims), _ptr(status), _stream(dev))
    _check(st, "pkv_copy_blocks")


def _host(t, name):
    if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_pinned():
        raise ValueError(f"{name} must be a pinned host tensor")
    return t


def swap_out(k_cache, v_cache, block_ids, host_k, host_v, k_scale=None, v_scale=None,
             host_k_scale=None, host_v_scale=None, status=None, kv_dtype=None):
    """Evict blocks to pinned host memory: host_k[i] := block block_ids[i] (likewise V
    and scales). Asynchronous on the current stream."""
    kv = _move_kv(k_cache, kv_dtype)
    dev, block, scale_block = _move_caches(kv, k_cache, v_cache, k_scale, v_scale)
    status = _status_word(status, dev)
    _require(block_ids, "block_ids", torch.int32, 1, dev)
    _host_buffers(kv, block_ids.numel(), block, scale_block, host_k, host_v, host_k_scale,
                  host_v_scale)
    dims = _move_dims(k_cache)
    with _OnDevice(dev):
        st = _lib().pkv_swap_out(_ptr(host_k), _ptr(host_v), _ptr(host_k_scale),
                                 _ptr(host_v_scale), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                 _ptr(v_scale), _ptr(block_ids), block_ids.numel(), kv,
                                 ctypes.byref(dims), _ptr(status), _stream(dev))
    _check(st, "pkv_swap_out")


def swap_in(k_cache, v_cache, block_ids, host_k, host_v, k_scale=None, v_scale=None,
            host_k_scale=None, host_v_scale=None, status=None, kv_dtype=None):
    """Bring evicted blocks back: block block_ids[i] := host_k[i] (likewise V and
    scales). Asynchronous on the current stream."""
    kv = _move_kv(k_cache, kv_dtype)
    dev, block, scale_block = _move_caches(kv, k_cache, v_cache, k_scale, v_scale)
    status = _status_word(status, dev)
    _require(block_ids, "block_ids", torch.int32, 1, dev)
    _host_buffers(kv, block_ids.numel(), block, scale_block, host_k, host_v, host_k_scale,
                  host_v_scale)
    dims = _move_dims(k_cache)
    with _OnDevice(dev):
        st = _lib().pkv_swap_in(_ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                _ptr(host_k), _ptr(host_v), _ptr(host_k_scale),
                                _ptr(host_v_scale), _ptr(block_ids), block_ids.numel(), kv,
                                ctypes.byref(dims), _ptr(status), _stream(dev))
    _check(st, "pkv_swap_in")


def multi_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                          num_blocks, max_blocks_per_seq, q_len, device=None):
    dims = Dims(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                max_blocks_per_seq)
    out = ctypes.c_size_t(0)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        st = _lib().pkv_decode_multi_workspace_bytes(ctypes.byref(dims), int(q_len),
                                                     ctypes.byref(out))
    _check(st, "pkv_decode_multi_workspace_bytes")
    return int(out.value)


def paged_decode_attention_multi(q, k_cache, v_cache, block_tables, context_lens, scale,
                                 out=None, workspace=None, status=None):
    """Attention for q_len new tokens per sequence in one call (speculative
    verification, q_len = k + 1, or a chunk of chunked prefill, q_len up to 256):
    q [B, q_len, Hq, D] bf16; the q_len newest tokens of
    every sequence are already in the bf16 caches and counted by ``context_lens``; new
    token i attends causally to positions 0 .. context_lens - q_len + i. Returns out
    [B, q_len, Hq, D] bf16."""
    dev = q.device
    status = _status_word(status, dev)
    _require(q, "q", torch.bfloat16, 4, dev)
    _require(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _require(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _require(block_tables, "block_tables", torch.int32, 2, dev)
    _require(context_lens, "context_lens", torch.int32, 1, dev)
    B, n, Hq, D = q.shape
    if k_cache.shape != v_cache.shape or k_cache.shape[3] != D:
        raise ValueError("cache shapes disagree with q")
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables / context_lens must have num_seqs rows")
    dims = _dims(B, Hq, k_cache, block_tables.shape[1])
    if out is None:
        out = torch.empty_like(q)
    else:
        _require(out, "out", torch.bfloat16, 4, dev)
        _same_shape(out, "out", q.shape)
    with _OnDevice(dev):
        need = ctypes.c_size_t(0)
        _check(_lib().pkv_decode_multi_workspace_bytes(ctypes.byref(dims), n,
                                                       ctypes.byref(need)),
               "pkv_decode_multi_workspace_bytes")
        workspace, ws_bytes = _workspace(workspace, need.value, dev)
        st = _lib().pkv_decode_multi_bf16(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                          _ptr(block_tables), _ptr(context_lens), n,
                                          float(scale), ctypes.byref(dims), _ptr(workspace),
                                          ws_bytes, _ptr(status), _stream(dev))
    _check(st, "pkv_decode_multi_bf16")
    return out


def multi_q8_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                             num_blocks, max_blocks_per_seq, q_len, kv_dtype, device=None):
    """Workspace of :func:`paged_decode_attention_multi_q8` (kv_dtype KV_INT8,
    KV_FP8_E4M3 or KV_FP8_E5M2)."""
    dims = Dims(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                max_blocks_per_seq)
    out = ctypes.c_size_t(0)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        st = _lib().pkv_decode_multi_q8_workspace_bytes(ctypes.byref(dims), int(q_len),
                                                        int(kv_dtype), ctypes.byref(out))
    _check(st, "pkv_decode_multi_q8_workspace_bytes")
    return int(out.value)


def _q8_kind(k_cache, fmt):
    """KV dtype code of a one-byte cache: int8 codes, or FP8 codes (uint8 with ``fmt``,
    or a torch float8 dtype)."""
    if k_cache.dtype == torch.int8:
        return KV_INT8
    if k_cache.dtype == torch.float8_e4m3fn:
        return KV_FP8_E4M3
    if k_cache.dtype == torch.float8_e5m2:
        return KV_FP8_E5M2
    if k_cache.dtype == torch.uint8:
        return _fp8_format(fmt)
    raise TypeError(f"a one-byte cache holds int8, uint8 or float8 codes, not {k_cache.dtype}")


def paged_decode_attention_multi_q8(q, k_cache, v_cache, k_scale, v_scale, block_tables,
                                    context_lens, scale, fmt="e5m2", out=None, workspace=None,
                                    status=None):
    """:func:`paged_decode_attention_multi` over a one-byte cache: int8 codes (INT8), or
    FP8 codes (uint8 with ``fmt`` "e4m3" / "e5m2", or the matching torch float8 dtype),
    with per-(token, KV head) fp32 scales ``k_scale``/``v_scale`` [NB, Hkv, bs]."""
    dev = q.device
    status = _status_word(status, dev)
    kv = _q8_kind(k_cache, fmt)
    _require(q, "q", torch.bfloat16, 4, dev)
    _require_any(k_cache, "k_cache", _code_dtypes(kv), 4, dev)
    _require_any(v_cache, "v_cache", _code_dtypes(kv), 4, dev)
    _require(k_scale, "k_scale", torch.float32, 3, dev)
    _require(v_scale, "v_scale", torch.float32, 3, dev)
    _require(block_tables, "block_tables", torch.int32, 2, dev)
    _require(context_lens, "context_lens", torch.int32, 1, dev)
    B, n, Hq, D = q.shape
    if k_cache.shape != v_cache.shape or k_cache.shape[3] != D:
        raise ValueError("cache shapes disagree with q")
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables / context_lens must have num_seqs rows")
    _cache_shapes(k_cache, v_cache, k_scale, v_scale)
    dims = _dims(B, Hq, k_cache, block_tables.shape[1])
    if out is None:
        out = torch.empty_like(q)
    else:
        _require(out, "out", torch.bfloat16, 4, dev)
        _same_shape(out, "out", q.shape)
    with _OnDevice(dev):
        need = ctypes.c_size_t(0)
        _check(_lib().pkv_decode_multi_q8_workspace_bytes(ctypes.byref(dims), n, kv,
                                                          ctypes.byref(need)),
               "pkv_decode_multi_q8_workspace_bytes")
        workspace, ws_bytes = _workspace(workspace, need.value, dev)
        st = _lib().pkv_decode_multi_q8(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(k_scale), _ptr(v_scale), _ptr(block_tables),
                                        _ptr(context_lens), n, float(scale), kv,
                                        ctypes.byref(dims), _ptr(workspace), ws_bytes,
                                        _ptr(status), _stream(dev))
    _check(st, "pkv_decode_multi_q8")
    return out


def cascade_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                            num_blocks, max_blocks_per_seq, prefix_blocks, device=None):
    dims = Dims(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                max_blocks_per_seq)
    out = ctypes.c_size_t(0)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        st = _lib().pkv_decode_cascade_workspace_bytes(ctypes.byref(dims), int(prefix_blocks),
                                                       ctypes.byref(out))
    _check(st, "pkv_decode_cascade_workspace_bytes")
    return int(out.value)


def paged_decode_attention_cascade(q, k_cache, v_cache, block_tables, context_lens,
                                   prefix_blocks, scale, out=None, workspace=None, status=None):
    """Decode attention for a batch whose tables all start with the same
    ``prefix_blocks`` physical blocks (row 0's): the shared prefix is attended once
    per KV head for every query row as a dense tensor-core contraction, the suffixes by
    the ordinary decode. Same result as :func:`paged_decode_attention` (bf16 caches)."""
    dev = q.device
    status = _status_word(status, dev)
    _require(q, "q", torch.bfloat16, 3, dev)
    _require(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _require(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _require(block_tables, "block_tables", torch.int32, 2, dev)
    _require(context_lens, "context_lens", torch.int32, 1, dev)
    B, Hq, D = q.shape
    if k_cache.shape != v_cache.shape or k_cache.shape[3] != D:
        raise ValueError("cache shapes disagree with q")
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables / context_lens must have num_seqs rows")
    dims = _dims(B, Hq, k_cache, block_tables.shape[1])
    if out is None:
        out = torch.empty_like(q)
    else:
        _require(out, "out", torch.bfloat16, 3, dev)
        _same_shape(out, "out", q.shape)
    with _OnDevice(dev):
        need = ctypes.c_size_t(0)
        _check(_lib().pkv_decode_cascade_workspace_bytes(ctypes.byref(dims), int(prefix_blocks),
                                                         ctypes.byref(need)),
               "pkv_decode_cascade_workspace_bytes")
        workspace, ws_bytes = _workspace(workspace, need.value, dev)
        st = _lib().pkv_decode_cascade_bf16(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                            _ptr(block_tables), _ptr(context_lens),
                                            int(prefix_blocks), float(scale), ctypes.byref(dims),
                                            _ptr(workspace), ws_bytes, _ptr(status),
                                            _stream(dev))
    _check(st, "pkv_decode_cascade_bf16")
    return out

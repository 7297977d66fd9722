"""Thin ctypes binding of ``include/lora.h`` (argument marshalling only).

Every function has the name of the C entry point it calls.  Device arguments
are CUDA torch tensors (their data pointers are passed), host arrays for
``lora_pool_load`` are numpy arrays or CPU tensors, and ``stream`` defaults to
torch's current stream.  A non-zero status raises :class:`LoraError`.  All
arithmetic happens in the CUDA library; importing this module fails when the
library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

LORA_OK = 0
LORA_ERR_ARG = -1
LORA_ERR_POOL_FULL = -2
LORA_ERR_RANK = -3
LORA_ERR_NOT_LOADED = -4
LORA_ERR_CUDA = -5
LORA_ERR_DEVICE_INDEX = -6
LORA_ERR_SHAPE = -7

LORA_F32 = 0
LORA_BF16 = 1

LORA_DEV_BAD_ADAPTER = 1
LORA_DEV_BAD_SEGMENTS = 2
LORA_DEV_WAIT_TIMEOUT = 4

LORA_NOALLOC_SCRATCH_BYTES = 16 << 20

LORA_TIER_GPU = 0
LORA_TIER_HOST = 1
LORA_TIER_DISK = 2

EXPORTS = ["lora_pool_create", "lora_pool_destroy", "lora_pool_load", "lora_pool_unload",
           "lora_pool_free_pages", "lora_sgmv_shrink", "lora_sgmv_expand", "lora_bgmv",
           "lora_layer_forward_workspace_size", "lora_layer_forward", "lora_get_error", "lora_strerror",
           "lora_launch_count", "lora_layer_forward_noalloc", "lora_tier_cache_create", "lora_tier_cache_destroy",
           "lora_tier_cache_touch", "lora_tier_cache_resident", "lora_tier_sim", "lora_pool_load_async",
           "lora_pool_unload_async", "lora_pool_prefetch", "lora_quantize_e4m3",
           "lora_layer_forward_fp8_workspace_size", "lora_layer_forward_fp8"]

if not os.path.exists(_build.LIB):
    raise ImportError(f"CUDA library {_build.LIB} is not built: run segmented_gathered_rank_gb300.build.build()")

LIB_PATH = _build.LIB
_lib = ctypes.CDLL(LIB_PATH)

_P = ctypes.c_void_p
_I = ctypes.c_int


def _sig(name, res, *args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = list(args)
    return f


_sig("lora_pool_create", _I, ctypes.POINTER(_P), _I, _I, _I, _I, _I, _I)
_sig("lora_pool_destroy", _I, _P)
_sig("lora_pool_load", _I, _P, _I, _I, _I, ctypes.c_float, _I, _I, _P, _P, _P)
_sig("lora_pool_unload", _I, _P, _I, _I)
_sig("lora_pool_free_pages", _I, _P)
_sig("lora_sgmv_shrink", _I, _P, _I, _P, _P, _I, _P, _P, _I, _I, _P)
_sig("lora_sgmv_expand", _I, _P, _I, _P, _I, _P, _P, _P, _I, _I, _P)
_sig("lora_bgmv", _I, _P, _I, _P, _P, _P, _I, _P)
_sig("lora_layer_forward_workspace_size", ctypes.c_size_t, _P, _I, _I, _I)
_sig("lora_layer_forward", _I, _P, _I, _P, _P, _P, _P, _P, _I, _I, _P, ctypes.c_size_t, _P)
_sig("lora_layer_forward_noalloc", _I, _P, _I, _P, _P, _P, _P, _P, _I, _I, _P)
_sig("lora_get_error", _I, _P, ctypes.POINTER(_I))
_sig("lora_strerror", ctypes.c_char_p, _I)
_sig("lora_launch_count", ctypes.c_ulonglong)


class AdapterSrc(ctypes.Structure):
    """``lora_adapter_src``: one entry of a prefetch list."""
    _fields_ = [("adapter", _I), ("matrix", _I), ("rank", _I), ("scale", ctypes.c_float), ("h_in", _I),
                ("h_out", _I), ("A_T", _P), ("B", _P)]


_sig("lora_pool_load_async", _I, _P, _I, _I, _I, ctypes.c_float, _I, _I, _P, _P, _P)
_sig("lora_pool_unload_async", _I, _P, _I, _I, _P)
_sig("lora_pool_prefetch", _I, _P, ctypes.POINTER(AdapterSrc), _I, _P)
_sig("lora_quantize_e4m3", _I, _P, _I, _I, _P, _P, _P)
_sig("lora_layer_forward_fp8_workspace_size", ctypes.c_size_t, _P, _I, _I, _I)
_sig("lora_layer_forward_fp8", _I, _P, _I, _P, _P, ctypes.c_float, _P, _P, _P, _I, _I, _P, ctypes.c_size_t, _P)
_sig("lora_tier_cache_create", _I, ctypes.POINTER(_P), _I, _I, _I)
_sig("lora_tier_cache_destroy", _I, _P)
_sig("lora_tier_cache_touch", _I, _P, _I, ctypes.POINTER(_I))
_sig("lora_tier_cache_resident", _I, _P, _I)
_sig("lora_tier_sim", _I, _P, ctypes.c_longlong, _I, _I, _I, ctypes.POINTER(ctypes.c_longlong))


class LoraError(RuntimeError):
    def __init__(self, status: int, where: str, device_status: int = 0):
        self.status = status
        self.device_status = device_status
        msg = f"{where}: {lora_strerror(status)} ({status})"
        if device_status:
            msg += f", device status 0x{device_status:x}"
        super().__init__(msg)


def _check(rc: int, where: str):
    if rc != LORA_OK:
        raise LoraError(rc, where)


def _dptr(t):
    """Device pointer of a CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _hptr(a):
    """Host pointer of a numpy array or CPU tensor (kept alive by the caller)."""
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        if not a.flags.c_contiguous:
            raise ValueError("expected a C-contiguous host array")
        return ctypes.c_void_p(a.ctypes.data)
    if a.is_cuda or not a.is_contiguous():
        raise ValueError("expected a contiguous CPU tensor")
    return ctypes.c_void_p(a.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def lora_strerror(status: int) -> str:
    return _lib.lora_strerror(int(status)).decode()


def lora_launch_count() -> int:
    return int(_lib.lora_launch_count())


def lora_pool_create(dtype: int, page_elems: int, n_pages: int, max_rank: int, n_matrices: int,
                     max_adapters: int) -> int:
    """Returns the pool handle (an opaque address)."""
    h = ctypes.c_void_p()
    _check(_lib.lora_pool_create(ctypes.byref(h), dtype, page_elems, n_pages, max_rank, n_matrices,
                                 max_adapters), "lora_pool_create")
    return h.value


def lora_pool_destroy(pool) -> None:
    _check(_lib.lora_pool_destroy(pool), "lora_pool_destroy")


def lora_pool_load(pool, adapter: int, matrix: int, rank: int, scale: float, h_in: int, h_out: int,
                   A_T, B, stream=None) -> None:
    _check(_lib.lora_pool_load(pool, adapter, matrix, rank, float(scale), h_in, h_out, _hptr(A_T), _hptr(B),
                               _stream(stream)), "lora_pool_load")


def lora_pool_unload(pool, adapter: int, matrix: int) -> None:
    _check(_lib.lora_pool_unload(pool, adapter, matrix), "lora_pool_unload")


def lora_pool_load_async(pool, adapter: int, matrix: int, rank: int, scale: float, h_in: int, h_out: int,
                         A_T, B, stream=None) -> None:
    """Enqueue an upload on ``stream`` and return (the host arrays are copied
    before the call returns)."""
    _check(_lib.lora_pool_load_async(pool, adapter, matrix, rank, float(scale), h_in, h_out, _hptr(A_T), _hptr(B),
                                     _stream(stream)), "lora_pool_load_async")


def lora_pool_unload_async(pool, adapter: int, matrix: int, stream=None) -> None:
    _check(_lib.lora_pool_unload_async(pool, adapter, matrix, _stream(stream)), "lora_pool_unload_async")


def lora_pool_prefetch(pool, entries, stream=None) -> int:
    """Upload every (adapter, matrix, rank, scale, h_in, h_out, A_T, B) entry not
    resident yet; returns how many uploads were enqueued."""
    entries = list(entries)
    arr = (AdapterSrc * max(1, len(entries)))()
    for i, (a, m, r, sc, hi, ho, at, b) in enumerate(entries):
        arr[i] = AdapterSrc(a, m, r, float(sc), hi, ho, _hptr(at), _hptr(b))
    rc = _lib.lora_pool_prefetch(pool, arr, len(entries), _stream(stream))
    if rc < 0:
        raise LoraError(rc, "lora_pool_prefetch")
    return int(rc)


def lora_pool_free_pages(pool) -> int:
    return int(_lib.lora_pool_free_pages(pool))


def lora_sgmv_shrink(pool, matrix, x, v, ld_v, seg_starts, seg_adapter, S, T, stream=None) -> None:
    _check(_lib.lora_sgmv_shrink(pool, matrix, _dptr(x), _dptr(v), ld_v, _dptr(seg_starts), _dptr(seg_adapter),
                                 S, T, _stream(stream)), "lora_sgmv_shrink")


def lora_sgmv_expand(pool, matrix, v, ld_v, y, seg_starts, seg_adapter, S, T, stream=None) -> None:
    _check(_lib.lora_sgmv_expand(pool, matrix, _dptr(v), ld_v, _dptr(y), _dptr(seg_starts), _dptr(seg_adapter),
                                 S, T, _stream(stream)), "lora_sgmv_expand")


def lora_bgmv(pool, matrix, x, y, token_adapter, T, stream=None) -> None:
    _check(_lib.lora_bgmv(pool, matrix, _dptr(x), _dptr(y), _dptr(token_adapter), T, _stream(stream)),
           "lora_bgmv")


def lora_layer_forward_workspace_size(pool, matrix, S, T) -> int:
    return int(_lib.lora_layer_forward_workspace_size(pool, matrix, S, T))


def lora_layer_forward(pool, matrix, x, W, y, seg_starts, seg_adapter, S, T, workspace, ws_bytes=None,
                       stream=None) -> None:
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib.lora_layer_forward(pool, matrix, _dptr(x), _dptr(W), _dptr(y), _dptr(seg_starts),
                                   _dptr(seg_adapter), S, T, _dptr(workspace), ws_bytes, _stream(stream)),
           "lora_layer_forward")


def lora_layer_forward_noalloc(pool, matrix, x, W, y, seg_starts, seg_adapter, S, T, stream=None) -> None:
    """lora_layer_forward with the library's fixed scratch instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    _check(_lib.lora_layer_forward_noalloc(pool, matrix, _dptr(x), _dptr(W), _dptr(y), _dptr(seg_starts),
                                           _dptr(seg_adapter), S, T, _stream(stream)),
           "lora_layer_forward_noalloc")


def lora_get_error(pool) -> tuple[int, int]:
    """(status, device status word); the word is cleared."""
    word = ctypes.c_int(0)
    rc = _lib.lora_get_error(pool, ctypes.byref(word))
    return int(rc), int(word.value)


def lora_tier_cache_create(n_keys: int, gpu_slots: int, host_slots: int) -> int:
    """Two-tier LRU residency cache (host only); returns its handle."""
    h = ctypes.c_void_p()
    _check(_lib.lora_tier_cache_create(ctypes.byref(h), n_keys, gpu_slots, host_slots), "lora_tier_cache_create")
    return h.value


def lora_tier_cache_destroy(cache) -> None:
    _check(_lib.lora_tier_cache_destroy(cache), "lora_tier_cache_destroy")


def lora_tier_cache_touch(cache, adapter: int) -> tuple[int, int]:
    """(tier that served the request, adapter the GPU tier evicted or -1)."""
    ev = ctypes.c_int(-1)
    rc = _lib.lora_tier_cache_touch(cache, adapter, ctypes.byref(ev))
    if rc < 0:
        raise LoraError(rc, "lora_tier_cache_touch")
    return int(rc), int(ev.value)


def lora_tier_cache_resident(cache, adapter: int) -> int:
    rc = _lib.lora_tier_cache_resident(cache, adapter)
    if rc < 0:
        raise LoraError(rc, "lora_tier_cache_resident")
    return int(rc)


def lora_tier_sim(trace, n_keys: int, gpu_slots: int, host_slots: int) -> tuple[int, int, int]:
    """(GPU hits, host hits, disk loads) of a request trace (int32 host array)."""
    tr = np.ascontiguousarray(trace, np.int32)
    counts = (ctypes.c_longlong * 3)()
    _check(_lib.lora_tier_sim(ctypes.c_void_p(tr.ctypes.data), len(tr), n_keys, gpu_slots, host_slots, counts),
           "lora_tier_sim")
    return int(counts[0]), int(counts[1]), int(counts[2])


def lora_quantize_e4m3(x, T, h, q, sx, stream=None) -> None:
    """Per-row e4m3 codes (uint8 tensor) and fp32 scales of a bf16 tensor."""
    _check(_lib.lora_quantize_e4m3(_dptr(x), T, h, _dptr(q), _dptr(sx), _stream(stream)), "lora_quantize_e4m3")


def lora_layer_forward_fp8_workspace_size(pool, matrix, S, T) -> int:
    return int(_lib.lora_layer_forward_fp8_workspace_size(pool, matrix, S, T))


def lora_layer_forward_fp8(pool, matrix, x, W8, w_scale, y, seg_starts, seg_adapter, S, T, workspace, ws_bytes=None,
                           stream=None) -> None:
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib.lora_layer_forward_fp8(pool, matrix, _dptr(x), _dptr(W8), float(w_scale), _dptr(y),
                                       _dptr(seg_starts), _dptr(seg_adapter), S, T, _dptr(workspace), ws_bytes,
                                       _stream(stream)), "lora_layer_forward_fp8")

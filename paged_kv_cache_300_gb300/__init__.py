"""Paged-attention forward for GB300: thin Python binding of libpa300.so.

Each function marshals torch tensors into the C ABI declared in
``include/pa.h`` (device pointers, sizes, the current CUDA stream) and
raises on a non-zero status.  All computation happens in the library's
CUDA kernels; there is no Python or CPU fallback: if the library is not
built, or no GPU is present, calls raise.

    pa_decode        decode step: in-place append + attention, one query per
                     sequence, through block_table
    pa_decode_contiguous  the same step over a contiguous cache (no table):
                     the twin that measures what paging costs
    pa_cache_update  scatter a packed varlen chunk into the paged pool
                     (optionally gather prefix + chunk into packed k/v)
    pa_varlen        packed variable-length attention (bf16: tcgen05)
    pa_varlen_paged  the same, reading keys through block_table from the pool
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "PAError", "library_path", "load", "pa_decode", "pa_decode_static_scratch",
    "pa_decode_contiguous", "pa_decode_contiguous_workspace_size",
    "pa_cache_update", "pa_varlen", "pa_varlen_paged",
    "pa_decode_workspace_size", "pa_status_string", "pa_version", "DEVERR_BAD_BLOCK",
    "DEVERR_OVERFLOW", "DEVERR_BAD_CU", "DEVERR_TIMEOUT",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "libpa300.so")

PA_F32, PA_BF16 = 0, 1
DEVERR_BAD_BLOCK, DEVERR_OVERFLOW, DEVERR_BAD_CU, DEVERR_TIMEOUT = 1, 2, 4, 8

_lock = threading.Lock()
_lib = None
_workspaces: dict = {}


class PAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: status {status} ({pa_status_string(status)})")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libpa300.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build the CUDA library first "
                "(python -m paged_kv_cache_300_gb300._build)")
        lib = ctypes.CDLL(_LIB_PATH)
        p, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.pa_decode_workspace_size.argtypes = [i] * 5 + [i]
        lib.pa_decode_workspace_size.restype = sz
        lib.pa_decode.argtypes = [p] * 8 + [i] * 7 + [i, f, p, sz, p, p]
        lib.pa_decode.restype = i
        lib.pa_decode_static_scratch.argtypes = [p] * 8 + [i] * 7 + [f, p, p]
        lib.pa_decode_static_scratch.restype = i
        lib.pa_decode_contiguous_workspace_size.argtypes = [i] * 4
        lib.pa_decode_contiguous_workspace_size.restype = sz
        lib.pa_decode_contiguous.argtypes = [p] * 7 + [i] * 5 + [f, p, sz, p, p]
        lib.pa_decode_contiguous.restype = i
        lib.pa_cache_update.argtypes = [p] * 10 + [i] * 8 + [i, p, p]
        lib.pa_cache_update.restype = i
        lib.pa_varlen.argtypes = [p] * 5 + [i] * 3 + [p] + [i] * 6 + [i, f, p, p]
        lib.pa_varlen.restype = i
        lib.pa_varlen_paged.argtypes = [p] * 6 + [i] * 3 + [p] + [i] * 8 + [i, f, p, p]
        lib.pa_varlen_paged.restype = i
        lib.pa_status_string.argtypes = [i]
        lib.pa_status_string.restype = ctypes.c_char_p
        lib.pa_version.argtypes = []
        lib.pa_version.restype = i
        _lib = lib
        return lib


def pa_status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()


def pa_version() -> int:
    return int(load().pa_version())


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return PA_BF16
    if t.dtype == torch.float32:
        return PA_F32
    raise TypeError(f"element tensors must be bfloat16 or float32, got {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_dev(*ts):
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("all tensors must live on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError("all tensors must be on the same device")
    return dev


def _check_host_or_dev(dev, *ts):
    """Per-step tensors of pa_decode: on `dev`, or page-locked host memory
    (which the kernel reads and writes in place over NVLink-C2C)."""
    for t in ts:
        if t is None:
            continue
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
        if t.is_cuda:
            if t.device != dev:
                raise ValueError("all tensors must be on the same device")
        elif not t.is_pinned():
            raise ValueError("host tensors must be page-locked (pin_memory())")


def _i32(t, name):
    if t is not None and t.dtype != torch.int32:
        raise TypeError(f"{name} must be int32")


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _call(name, rc):
    if rc != 0:
        raise PAError(name, rc)


def pa_decode_workspace_size(batch, num_heads, num_kv_heads, head_dim, block_size,
                             dtype=torch.bfloat16) -> int:
    dt = PA_BF16 if dtype == torch.bfloat16 else PA_F32
    return int(load().pa_decode_workspace_size(batch, num_heads, num_kv_heads, head_dim,
                                               block_size, dt))


def _workspace(dev, nbytes):
    if nbytes == 0:
        return None
    key = (dev.index, torch.cuda.current_stream(dev).cuda_stream)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)  # zero on first use
        _workspaces[key] = ws
    return ws


def pa_decode(q, k_cache, v_cache, block_table, cache_seqlens, k_new, v_new, out=None,
              softmax_scale: float = 0.0, workspace=None, dev_err=None, stream=None):
    """Decode step (see include/pa.h).  q [B, Hq, D]; k_cache/v_cache
    [NB, bs, Hkv, D] (the new token is written in place); block_table
    [B, MB] int32; cache_seqlens [B] int32; k_new/v_new [B, Hkv, D].
    Returns out [B, Hq, D].  q, block_table, cache_seqlens, k_new, v_new
    and out may be pinned host tensors (read and written in place; `out`
    defaults to a pinned host tensor then); the pools, workspace and
    dev_err live on the GPU."""
    dev = _check_dev(k_cache, v_cache, workspace, dev_err)
    _check_host_or_dev(dev, q, block_table, cache_seqlens, k_new, v_new, out)
    _i32(block_table, "block_table")
    _i32(cache_seqlens, "cache_seqlens")
    _i32(dev_err, "dev_err")
    dt = _dtype(q)
    for t in (k_cache, v_cache, k_new, v_new):
        if t.dtype != q.dtype:
            raise TypeError("q, k_cache, v_cache, k_new, v_new must share a dtype")
    b, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if d2 != d or v_cache.shape != k_cache.shape or k_new.shape != (b, hkv, d) or \
            v_new.shape != (b, hkv, d) or block_table.shape[0] != b or cache_seqlens.shape != (b,):
        raise ValueError("inconsistent shapes")
    mb = block_table.shape[1]
    if out is None:
        out = torch.empty_like(q, pin_memory=not q.is_cuda)
    elif out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("out must match q")
    lib = load()
    if workspace is None:
        workspace = _workspace(dev, int(lib.pa_decode_workspace_size(b, hq, hkv, d, bs, dt)))
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.pa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                       _ptr(cache_seqlens), _ptr(k_new), _ptr(v_new), _ptr(out), b, hq, hkv, d,
                       nb, bs, mb, dt, float(softmax_scale), _ptr(workspace), wbytes,
                       _ptr(dev_err), _stream(stream))
    _call("pa_decode", rc)
    return out


def pa_decode_static_scratch(q, k_cache, v_cache, block_table, cache_seqlens, k_new, v_new,
                             out=None, softmax_scale: float = 0.0, dev_err=None, stream=None):
    """pa_decode (bf16) with the library's built-in 16 MiB scratch instead
    of a workspace: for callers that cannot allocate device memory at call
    time.  Calls that may overlap on the GPU must be serialised."""
    _check_dev(q, k_cache, v_cache, block_table, cache_seqlens, k_new, v_new, out, dev_err)
    _i32(block_table, "block_table")
    _i32(cache_seqlens, "cache_seqlens")
    _i32(dev_err, "dev_err")
    if q.dtype != torch.bfloat16:
        raise TypeError("pa_decode_static_scratch takes bfloat16 tensors")
    b, hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    rc = load().pa_decode_static_scratch(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                         _ptr(cache_seqlens), _ptr(k_new), _ptr(v_new), _ptr(out),
                                         b, hq, hkv, d, nb, bs, block_table.shape[1],
                                         float(softmax_scale), _ptr(dev_err), _stream(stream))
    _call("pa_decode_static_scratch", rc)
    return out


def pa_decode_contiguous_workspace_size(batch, num_heads, num_kv_heads, head_dim) -> int:
    return int(load().pa_decode_contiguous_workspace_size(batch, num_heads, num_kv_heads,
                                                          head_dim))


def pa_decode_contiguous(q, k_cache, v_cache, cache_seqlens, k_new, v_new, out=None,
                         softmax_scale: float = 0.0, workspace=None, dev_err=None, stream=None):
    """Decode step over a contiguous cache (see include/pa.h): q [B, Hq, D];
    k_cache/v_cache [B, max_seqlen, Hkv, D] (the new token is written in
    place at [b, cache_seqlens[b]]); k_new/v_new [B, Hkv, D].  bf16 only.
    Returns out [B, Hq, D]."""
    dev = _check_dev(q, k_cache, v_cache, cache_seqlens, k_new, v_new, out, workspace, dev_err)
    _i32(cache_seqlens, "cache_seqlens")
    _i32(dev_err, "dev_err")
    if q.dtype != torch.bfloat16:
        raise TypeError("pa_decode_contiguous takes bfloat16 tensors")
    for t in (k_cache, v_cache, k_new, v_new):
        if t.dtype != q.dtype:
            raise TypeError("q, k_cache, v_cache, k_new, v_new must share a dtype")
    b, hq, d = q.shape
    b2, lmax, hkv, d2 = k_cache.shape
    if b2 != b or d2 != d or v_cache.shape != k_cache.shape or k_new.shape != (b, hkv, d) or \
            v_new.shape != (b, hkv, d) or cache_seqlens.shape != (b,):
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("out must match q")
    lib = load()
    if workspace is None:
        workspace = _workspace(dev, int(lib.pa_decode_contiguous_workspace_size(b, hq, hkv, d)))
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.pa_decode_contiguous(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cache_seqlens),
                                  _ptr(k_new), _ptr(v_new), _ptr(out), b, hq, hkv, d, lmax,
                                  float(softmax_scale), _ptr(workspace), wbytes, _ptr(dev_err),
                                  _stream(stream))
    _call("pa_decode_contiguous", rc)
    return out


def pa_cache_update(k_chunk, v_chunk, cu_seq_lens_q, cache_seqlens, block_table, k_cache,
                    v_cache, k_full=None, v_full=None, cu_seq_lens_k=None, dev_err=None,
                    stream=None):
    """Scatter the packed chunk [Tq, Hkv, D] into the pool at positions
    cache_seqlens[b] + i; with k_full/v_full/cu_seq_lens_k also gather each
    request's prefix + chunk into the packed [Tk, Hkv, D] tensors."""
    _check_dev(k_chunk, v_chunk, cu_seq_lens_q, cache_seqlens, block_table, k_cache, v_cache,
               k_full, v_full, cu_seq_lens_k, dev_err)
    for t, n in ((cu_seq_lens_q, "cu_seq_lens_q"), (cache_seqlens, "cache_seqlens"),
                 (block_table, "block_table"), (cu_seq_lens_k, "cu_seq_lens_k"),
                 (dev_err, "dev_err")):
        _i32(t, n)
    dt = _dtype(k_cache)
    nb, bs, hkv, d = k_cache.shape
    b = cache_seqlens.shape[0]
    tq = k_chunk.shape[0]
    tk = 0 if k_full is None else k_full.shape[0]
    rc = load().pa_cache_update(_ptr(k_chunk), _ptr(v_chunk), _ptr(cu_seq_lens_q),
                                _ptr(cache_seqlens), _ptr(block_table), _ptr(k_cache),
                                _ptr(v_cache), _ptr(k_full), _ptr(v_full), _ptr(cu_seq_lens_k),
                                b, tq, tk, hkv, d, nb, bs, block_table.shape[1], dt,
                                _ptr(dev_err), _stream(stream))
    _call("pa_cache_update", rc)
    return k_full, v_full


def pa_varlen(q, k, v, cu_seq_lens_q, cu_seq_lens_k, max_length_q: int, max_length_k: int,
              causal: bool, out=None, softmax_scale: float = 0.0, dev_err=None, stream=None):
    """Varlen attention: q [Tq, Hq, D], k/v [Tk, Hkv, D] -> out [Tq, Hq, D]."""
    _check_dev(q, k, v, cu_seq_lens_q, cu_seq_lens_k, out, dev_err)
    _i32(cu_seq_lens_q, "cu_seq_lens_q")
    _i32(cu_seq_lens_k, "cu_seq_lens_k")
    dt = _dtype(q)
    tq, hq, d = q.shape
    tk, hkv, _ = k.shape
    if out is None:
        out = torch.empty_like(q)
    rc = load().pa_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seq_lens_q), _ptr(cu_seq_lens_k),
                          int(max_length_q), int(max_length_k), int(bool(causal)), _ptr(out),
                          cu_seq_lens_q.shape[0] - 1, tq, tk, hq, hkv, d, dt,
                          float(softmax_scale), _ptr(dev_err), _stream(stream))
    _call("pa_varlen", rc)
    return out


def pa_varlen_paged(q, k_cache, v_cache, block_table, cu_seq_lens_q, seqlens_k,
                    max_length_q: int, max_length_k: int, causal: bool, out=None,
                    softmax_scale: float = 0.0, dev_err=None, stream=None):
    """Varlen attention with keys read through block_table: q [Tq, Hq, D];
    k_cache/v_cache [NB, bs, Hkv, D]; block_table [B, MB]; seqlens_k [B]
    (keys of each request in the pool).  Returns out [Tq, Hq, D]."""
    _check_dev(q, k_cache, v_cache, block_table, cu_seq_lens_q, seqlens_k, out, dev_err)
    for t, n in ((block_table, "block_table"), (cu_seq_lens_q, "cu_seq_lens_q"),
                 (seqlens_k, "seqlens_k"), (dev_err, "dev_err")):
        _i32(t, n)
    dt = _dtype(q)
    tq, hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    rc = load().pa_varlen_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                _ptr(cu_seq_lens_q), _ptr(seqlens_k), int(max_length_q),
                                int(max_length_k), int(bool(causal)), _ptr(out),
                                cu_seq_lens_q.shape[0] - 1, tq, hq, hkv, d, nb, bs,
                                block_table.shape[1], dt, float(softmax_scale), _ptr(dev_err),
                                _stream(stream))
    _call("pa_varlen_paged", rc)
    return out

"""fp64 CPU oracle for paged-attention forward.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the library and its
binding never do.  It shares no code with the CUDA path.

``pa_oracle.c`` holds the plain loops (see its header for the passages each
function restates); this module compiles it with gcc (``build()``), loads it
with ctypes and exposes numpy-facing wrappers.  ``ref_np`` is a second,
independent numpy float64 route used for brute-force cross checks on tiny
inputs.

Parity status of each function (what pins it, in tests/test_oracle_*.py):
  decode          pinned: the decode worked example of "Perhatian berhalaman"
                  (append slots), the scalar-head example of "PagedAttention"
                  (paweldubiel.com, output 3 under both placements), paged ==
                  contiguous, closed forms, brute force.
  cache_update    pinned: bitwise placement checks against hand-derived
                  positions, round trip with gather.
  varlen          pinned: the cu_seq_lens example of "Perhatian berhalaman"
                  (empty key set for r0), causal closed forms, brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libpa_oracle.so")
_lock = threading.Lock()
_handle = None

F32, BF16 = 0, 1

_ERRORS = {
    -1: "bad arguments",
    -2: "a needed block_table entry is not a valid block",
    -3: "position beyond max_blocks_per_seq * block_size",
    -4: "inconsistent cumulative lengths",
}


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into a shared library (gcc, OpenMP)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str):
    lib = ctypes.CDLL(path)
    p, i, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    lib.pa_oracle_decode.argtypes = [p] * 8 + [i] * 8 + [d, i]
    lib.pa_oracle_attend_contiguous.argtypes = [p, p, p, i, i, ctypes.c_int64, ctypes.c_int64,
                                                i, d, p]
    lib.pa_oracle_cache_update.argtypes = [p] * 10 + [i] * 7
    lib.pa_oracle_varlen.argtypes = [p] * 5 + [i] * 6 + [d, p, i]
    lib.pa_oracle_max_threads.argtypes = []
    for f in (lib.pa_oracle_decode, lib.pa_oracle_attend_contiguous, lib.pa_oracle_cache_update,
              lib.pa_oracle_varlen, lib.pa_oracle_max_threads):
        f.restype = ctypes.c_int
    return lib


def _lib():
    global _handle
    with _lock:
        if _handle is None:
            _handle = _bind(build())
    return _handle


def compile_variant(src_text: str, out_dir: str):
    """Compile an edited copy of the oracle source (used by the tests that
    plant a mistake in the oracle to show the pins catch it) and return a
    namespace with the same wrappers bound to it."""
    os.makedirs(out_dir, exist_ok=True)
    src = os.path.join(out_dir, "variant.c")
    so = os.path.join(out_dir, "libvariant.so")
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c99", src, "-o", so,
                    "-lm"], check=True)
    return _Bound(_bind(so))


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def max_threads() -> int:
    return int(_lib().pa_oracle_max_threads())


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:  # bfloat16 bit patterns
        return BF16
    raise TypeError(f"oracle takes float32 or bfloat16 bits (uint16), got {a.dtype}")


def _c(a):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int):
    if rc != 0:
        raise OracleError(_ERRORS.get(rc, f"oracle error {rc}"))


def decode(q, k_cache, v_cache, block_table, cache_seqlens, k_new, v_new,
           softmax_scale: float = 0.0, nthreads: int = 0, _l=None) -> np.ndarray:
    """Decode step; k_cache/v_cache are modified in place (the append).

    q [B, Hq, D]; k_cache/v_cache [NB, bs, Hkv, D]; block_table [B, MB] int32;
    cache_seqlens [B] int32; k_new/v_new [B, Hkv, D].  Returns out [B, Hq, D]
    float64.  Element arrays are float32 or bfloat16 bit patterns (uint16).
    """
    dt = _dtype_code(q)
    b, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    assert d2 == d and v_cache.shape == k_cache.shape
    mb = block_table.shape[1]
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(cache_seqlens, dtype=np.int32)
    out = np.zeros((b, hq, d), dtype=np.float64)
    rc = (_l or _lib()).pa_oracle_decode(_c(q), _c(k_cache), _c(v_cache), _c(bt), _c(sl), _c(k_new),
                                 _c(v_new), _c(out), b, hq, hkv, d, nb, bs, mb, dt,
                                 float(softmax_scale), int(nthreads))
    _check(rc)
    return out


def attend_contiguous(q_row, k_rows, v_rows, head: int = 0, softmax_scale: float = 0.0, _l=None):
    """One query row [D] against contiguous k/v [n, Hkv, D] of kv head `head`."""
    dt = _dtype_code(q_row)
    n, hkv, d = k_rows.shape
    out = np.zeros(d, dtype=np.float64)
    _check((_l or _lib()).pa_oracle_attend_contiguous(_c(q_row), _c(k_rows), _c(v_rows), n, d,
                                              hkv * d, head * d, dt, float(softmax_scale),
                                              _c(out)))
    return out


def cache_update(k_chunk, v_chunk, cu_seq_lens_q, prefix_lens, block_table, k_cache, v_cache,
                 cu_seq_lens_k=None, _l=None):
    """Scatter a packed chunk into the pool (in place); with cu_seq_lens_k,
    also return the gathered (k_full, v_full) [total_k, Hkv, D]."""
    dt = _dtype_code(k_chunk)
    nb, bs, hkv, d = k_cache.shape
    b = len(prefix_lens)
    mb = block_table.shape[1]
    cq = np.ascontiguousarray(cu_seq_lens_q, dtype=np.int32)
    pl = np.ascontiguousarray(prefix_lens, dtype=np.int32)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    kf = vf = None
    ck = None
    if cu_seq_lens_k is not None:
        ck = np.ascontiguousarray(cu_seq_lens_k, dtype=np.int32)
        kf = np.zeros((int(ck[-1]), hkv, d), dtype=k_chunk.dtype)
        vf = np.zeros_like(kf)
    rc = (_l or _lib()).pa_oracle_cache_update(
        _c(k_chunk), _c(v_chunk), _c(cq), _c(pl), _c(bt), _c(k_cache), _c(v_cache),
        None if kf is None else _c(kf), None if vf is None else _c(vf),
        None if ck is None else _c(ck), b, hkv, d, nb, bs, mb, dt)
    _check(rc)
    return kf, vf


def varlen(q, k, v, cu_seq_lens_q, cu_seq_lens_k, causal: bool, softmax_scale: float = 0.0,
           nthreads: int = 0, _l=None) -> np.ndarray:
    """Varlen attention; q [Tq, Hq, D], k/v [Tk, Hkv, D] -> out [Tq, Hq, D] float64."""
    dt = _dtype_code(q)
    tq, hq, d = q.shape
    tk, hkv, _ = k.shape
    cq = np.ascontiguousarray(cu_seq_lens_q, dtype=np.int32)
    ck = np.ascontiguousarray(cu_seq_lens_k, dtype=np.int32)
    b = len(cq) - 1
    out = np.zeros((tq, hq, d), dtype=np.float64)
    _check((_l or _lib()).pa_oracle_varlen(_c(q), _c(k), _c(v), _c(cq), _c(ck), b, hq, hkv, d,
                                   int(bool(causal)), dt, float(softmax_scale), _c(out),
                                   int(nthreads)))
    return out


class _Bound:
    """The wrappers above bound to one compiled library."""

    def __init__(self, lib):
        self._l = lib

    def decode(self, *a, **k):
        return decode(*a, _l=self._l, **k)

    def attend_contiguous(self, *a, **k):
        return attend_contiguous(*a, _l=self._l, **k)

    def cache_update(self, *a, **k):
        return cache_update(*a, _l=self._l, **k)

    def varlen(self, *a, **k):
        return varlen(*a, _l=self._l, **k)

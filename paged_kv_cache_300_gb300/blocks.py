"""Host block manager of the paged KV pool (binding of include/pa_blocks.h).

Tracks which physical blocks each sequence holds (free list, reference
counts, shared full-block prefixes) and exports the block_table /
cache_seqlens arrays the attention calls read.  Host-only C++ in
libpa300.so; this module only marshals arguments.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import load

ERRORS = {-1: "bad arguments", -2: "unknown sequence", -3: "sequence id already in use",
          -4: "not enough free blocks", -5: "sequence would exceed max_blocks_per_seq"}


class BlockManagerError(RuntimeError):
    def __init__(self, what, code):
        super().__init__(f"{what}: {ERRORS.get(code, code)}")
        self.code = code


def _lib():
    lib = load()
    if not getattr(lib, "_pa_bm_bound", False):
        v, i, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        lib.pa_bm_create.argtypes = [i, i, i]
        lib.pa_bm_create.restype = v
        lib.pa_bm_destroy.argtypes = [v]
        lib.pa_bm_destroy.restype = None
        for f, args in (("pa_bm_add", [v, i64, i]), ("pa_bm_fork", [v, i64, i64, i]),
                        ("pa_bm_append", [v, i64, i]), ("pa_bm_free", [v, i64]),
                        ("pa_bm_num_free", [v]), ("pa_bm_refcount", [v, i]),
                        ("pa_bm_length", [v, i64]), ("pa_bm_tables", [v, v, i, v, v])):
            fn = getattr(lib, f)
            fn.argtypes = args
            fn.restype = i
        lib._pa_bm_bound = True
    return lib


class BlockManager:
    """Physical-block bookkeeping for a pool of `num_blocks` blocks."""

    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int):
        self._lib = _lib()
        self._h = self._lib.pa_bm_create(num_blocks, block_size, max_blocks_per_seq)
        if not self._h:
            raise BlockManagerError("create", -1)
        self.num_blocks, self.block_size, self.max_blocks_per_seq = (
            num_blocks, block_size, max_blocks_per_seq)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.pa_bm_destroy(h)
            self._h = None

    def _check(self, what, rc):
        if rc < 0:
            raise BlockManagerError(what, rc)
        return rc

    def add(self, seq_id: int, num_tokens: int):
        self._check("add", self._lib.pa_bm_add(self._h, seq_id, num_tokens))

    def fork(self, parent: int, child: int, shared_tokens: int):
        self._check("fork", self._lib.pa_bm_fork(self._h, parent, child, shared_tokens))

    def append(self, seq_id: int, num_tokens: int = 1):
        self._check("append", self._lib.pa_bm_append(self._h, seq_id, num_tokens))

    def free(self, seq_id: int):
        self._check("free", self._lib.pa_bm_free(self._h, seq_id))

    def num_free(self) -> int:
        return self._check("num_free", self._lib.pa_bm_num_free(self._h))

    def refcount(self, block: int) -> int:
        return self._check("refcount", self._lib.pa_bm_refcount(self._h, block))

    def length(self, seq_id: int) -> int:
        return self._check("length", self._lib.pa_bm_length(self._h, seq_id))

    def tables(self, seq_ids):
        """(block_table [n, max_blocks_per_seq] int32, lengths [n] int32),
        CPU tensors in the order of `seq_ids`."""
        ids = np.ascontiguousarray(np.asarray(list(seq_ids), dtype=np.int64))
        n = len(ids)
        table = np.empty((n, self.max_blocks_per_seq), dtype=np.int32)
        lengths = np.empty(n, dtype=np.int32)
        self._check("tables", self._lib.pa_bm_tables(
            self._h, ids.ctypes.data_as(ctypes.c_void_p), n,
            table.ctypes.data_as(ctypes.c_void_p), lengths.ctypes.data_as(ctypes.c_void_p)))
        return torch.from_numpy(table), torch.from_numpy(lengths)

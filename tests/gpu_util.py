"""Helpers shared by the GPU parity tests: run a workload through the C ABI
(via the binding) and through the oracle on the same bits, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_cache_300_gb300 as pa
from workloads import to_numpy

BF16_TOL = 1e-2  # abs and rel, per element, vs the fp64 oracle
F32_TOL = 1e-5


def tol_for(dtype):
    return BF16_TOL if dtype == torch.bfloat16 else F32_TOL


def assert_close(gpu: torch.Tensor, ref: np.ndarray, dtype, what=""):
    """|gpu - ref| <= tol + tol * |ref| element by element."""
    tol = tol_for(dtype)
    g = gpu.detach().float().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref)
    bound = tol + tol * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside tolerance "
            f"(max abs err {err.max():.3e}); first {idx.tolist()}")
    return float(err.max()), float((err / np.maximum(np.abs(ref), 1e-30)).max())


def gpu_decode(case, dev="cuda", dev_err=None):
    """Run pa_decode on copies of the case's tensors; return (out, k_pool, v_pool)."""
    t = lambda x: x.to(dev).contiguous()
    kc, vc = t(case.k_cache), t(case.v_cache)
    out = pa.pa_decode(t(case.q), kc, vc, t(case.block_table), t(case.cache_seqlens),
                       t(case.k_new), t(case.v_new), dev_err=dev_err)
    torch.cuda.synchronize()
    return out, kc, vc


def oracle_decode(case, rows=None):
    """Oracle on the case (optionally a subset of sequences); returns
    (out fp64, k_pool, v_pool) with the appends applied to numpy copies."""
    q, kn, vn = to_numpy(case.q), to_numpy(case.k_new), to_numpy(case.v_new)
    tab, sl = case.block_table.numpy(), case.cache_seqlens.numpy()
    if rows is not None:
        rows = np.asarray(rows)
        q, kn, vn = q[rows].copy(), kn[rows].copy(), vn[rows].copy()
        tab, sl = tab[rows].copy(), sl[rows].copy()
    kc, vc = to_numpy(case.k_cache).copy(), to_numpy(case.v_cache).copy()
    out = oracle.decode(np.ascontiguousarray(q), kc, vc, np.ascontiguousarray(tab),
                        np.ascontiguousarray(sl), np.ascontiguousarray(kn),
                        np.ascontiguousarray(vn))
    return out, kc, vc


def bits(t: torch.Tensor) -> np.ndarray:
    return to_numpy(t.cpu())

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


def assert_close(gpu: torch.Tensor, ref: np.ndarray, dtype, what="", discriminating=True):
    """|gpu - ref| <= tol * s + tol * |ref| element by element, with
    s = min(1, max|ref|): the pages' absolute-plus-relative bound, with the
    absolute part scaled down to the output's own size when the outputs are
    small, so that a comparison of tiny outputs still tests something.

    With `discriminating` (the default) the check also proves it can fail:
    an all-zero output must fall outside the bound somewhere, else the test
    itself is rejected (a case whose reference is all zeros passes False)."""
    tol = tol_for(dtype)
    g = gpu.detach().float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, f"{what}: shape {g.shape} vs {ref.shape}"
    assert np.isfinite(g).all(), f"{what}: non-finite values in the GPU output"
    scale = min(1.0, float(np.abs(ref).max())) if ref.size else 1.0
    err = np.abs(g - ref)
    bound = tol * scale + tol * np.abs(ref)
    if discriminating and ref.size:
        assert (np.abs(ref) > bound).any(), (
            f"{what}: the check cannot fail (an all-zero output would pass)")
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside tolerance "
            f"(max abs err {err.max():.3e}, max |ref| {np.abs(ref).max():.3e}); first "
            f"{idx.tolist()}")
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


def same_bits(a: np.ndarray, b: np.ndarray) -> bool:
    """Bitwise equality of two element arrays (NaN patterns included)."""
    if a.shape != b.shape or a.dtype.itemsize != b.dtype.itemsize:
        return False
    u = {2: np.uint16, 4: np.uint32, 8: np.uint64}[a.dtype.itemsize]
    return np.array_equal(np.ascontiguousarray(a).view(u), np.ascontiguousarray(b).view(u))

"""Second, independent float64 route (numpy), for brute force on tiny inputs.

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``).

Where ``pa_oracle.c`` walks the block table one token at a time in three
passes, this module first materialises the contiguous K/V of a sequence with
numpy fancy indexing and then evaluates softmax(q K^T * scale) V with matrix
products.  The two share no code, so agreement between them checks the
gather indexing and the arithmetic of both.

``merge_partials`` restates the partial merge of "39 · PagedAttention"
(inference-notes, section "3. Trên GPU"): two partial results with running
maximum m_i and exponential sum l_i combine as m = max(m1, m2),
l = l1·e^(m1−m) + l2·e^(m2−m).  The printed formula runs the two equations
together; the output accumulator is merged with the same weights, and a part
with m = −inf contributes nothing.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact upcast of bfloat16 bit patterns (uint16) to float64."""
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_f64(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return bf16_bits_to_f64(a)
    return a.astype(np.float64)


def gather_sequence(pool: np.ndarray, table_row: np.ndarray, length: int, block_size: int):
    """Contiguous [length, Hkv, D] rows of one sequence (logical order)."""
    pos = np.arange(length)
    phys = table_row[pos // block_size]
    assert (phys >= 0).all(), "needed block not allocated"
    return pool[phys, pos % block_size]


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, mask=None):
    """softmax(q k^T * scale) v for q [M, D], k/v [N, D]; all-masked rows -> 0."""
    s = (q @ k.T) * scale
    if mask is not None:
        s = np.where(mask, s, -np.inf)
    out = np.zeros((q.shape[0], v.shape[1]))
    for i in range(q.shape[0]):
        if not np.isfinite(s[i]).any():
            continue
        w = np.exp(s[i] - s[i].max())
        out[i] = (w / w.sum()) @ v
    return out


def decode(q, k_cache, v_cache, block_table, cache_seqlens, k_new, v_new, softmax_scale=0.0):
    """Same contract as ``oracle.decode`` (pools modified in place)."""
    b, hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    g = hq // hkv
    scale = softmax_scale if softmax_scale > 0 else 1.0 / np.sqrt(d)
    for i in range(b):
        pos = int(cache_seqlens[i])
        p = block_table[i, pos // bs]
        k_cache[p, pos % bs] = k_new[i]
        v_cache[p, pos % bs] = v_new[i]
    out = np.zeros((b, hq, d))
    for i in range(b):
        t = int(cache_seqlens[i]) + 1
        kk = to_f64(gather_sequence(k_cache, block_table[i], t, bs))
        vv = to_f64(gather_sequence(v_cache, block_table[i], t, bs))
        qq = to_f64(q[i])
        for h in range(hq):
            out[i, h] = attention(qq[h:h + 1], kk[:, h // g], vv[:, h // g], scale)[0]
    return out


def varlen(q, k, v, cu_q, cu_k, causal, softmax_scale=0.0):
    """Same contract as ``oracle.varlen``."""
    tq, hq, d = q.shape
    hkv = k.shape[1]
    g = hq // hkv
    scale = softmax_scale if softmax_scale > 0 else 1.0 / np.sqrt(d)
    out = np.zeros((tq, hq, d))
    qf, kf, vf = to_f64(q), to_f64(k), to_f64(v)
    for r in range(len(cu_q) - 1):
        q0, q1, k0, k1 = int(cu_q[r]), int(cu_q[r + 1]), int(cu_k[r]), int(cu_k[r + 1])
        ql, kl = q1 - q0, k1 - k0
        if ql == 0:
            continue
        mask = None
        if causal:
            mask = np.arange(kl)[None, :] <= (np.arange(ql)[:, None] + kl - ql)
        for h in range(hq):
            out[q0:q1, h] = attention(qf[q0:q1, h], kf[k0:k1, h // g], vf[k0:k1, h // g], scale,
                                      mask)
    return out


def partial(scores: np.ndarray, values: np.ndarray):
    """Unnormalised partial (m, l, acc) of one query over a subset of keys."""
    if scores.size == 0:
        return -np.inf, 0.0, np.zeros(values.shape[1])
    m = scores.max()
    e = np.exp(scores - m)
    return m, e.sum(), e @ values


def merge_partials(p1, p2):
    """m = max(m1, m2); l = l1 e^(m1-m) + l2 e^(m2-m); acc merged alike."""
    m1, l1, a1 = p1
    m2, l2, a2 = p2
    m = max(m1, m2)
    if m == -np.inf:
        return m, 0.0, np.zeros_like(a1)
    w1 = 0.0 if m1 == -np.inf else np.exp(m1 - m)
    w2 = 0.0 if m2 == -np.inf else np.exp(m2 - m)
    return m, l1 * w1 + l2 * w2, a1 * w1 + a2 * w2

"""Oracle vs an independent numpy float64 route, and planted mistakes.

The brute-force half runs both routes on tiny random inputs.  The second
half plants plausible mistakes in a copy of the oracle source (on the CPU)
and checks that the page-derived pins reject each one.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import ref_np
from tests.conftest import bf16_bits, load_golden


def _rand_decode(seed, dtype):
    rng = np.random.default_rng(seed)
    b = int(rng.integers(1, 4))
    hkv = int(rng.choice([1, 2]))
    g = int(rng.choice([1, 2, 3]))
    hq = hkv * g
    d = int(rng.choice([1, 4, 8]))
    bs = int(rng.choice([2, 4, 8]))
    lens = rng.integers(0, 40, size=b).astype(np.int32)
    need = -(-(lens + 1) // bs)
    nb = int(need.sum()) + 3
    perm = rng.permutation(nb)
    mb = int(need.max()) + 1
    table = np.full((b, mb), -1, np.int32)
    off = 0
    for i, n in enumerate(need):
        table[i, :n] = perm[off:off + n]
        off += n
    mk = lambda *s: rng.standard_normal(s).astype(np.float32) * 2
    arrs = [mk(b, hq, d), mk(nb, bs, hkv, d), mk(nb, bs, hkv, d), mk(b, hkv, d), mk(b, hkv, d)]
    if dtype == np.uint16:
        arrs = [bf16_bits(a) for a in arrs]
    return arrs, table, lens


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_decode_matches_numpy_route(seed, dtype):
    (q, kc, vc, kn, vn), table, lens = _rand_decode(seed, dtype)
    kc2, vc2 = kc.copy(), vc.copy()
    out = oracle.decode(q, kc, vc, table, lens, kn, vn)
    ref = ref_np.decode(q, kc2, vc2, table, lens, kn, vn)
    assert np.array_equal(kc, kc2) and np.array_equal(vc, vc2)  # same append, bitwise
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("seed", range(10))
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_matches_numpy_route(seed, causal):
    rng = np.random.default_rng(100 + seed)
    b = int(rng.integers(1, 4))
    ql = rng.integers(0, 12, size=b)
    kl = rng.integers(0, 15, size=b)
    hkv = int(rng.choice([1, 2]))
    hq = hkv * int(rng.choice([1, 2, 4]))
    d = int(rng.choice([2, 8]))
    cu_q = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(kl)]).astype(np.int32)
    q = rng.standard_normal((cu_q[-1], hq, d)).astype(np.float32)
    k = rng.standard_normal((cu_k[-1], hkv, d)).astype(np.float32)
    v = rng.standard_normal((cu_k[-1], hkv, d)).astype(np.float32)
    out = oracle.varlen(q, k, v, cu_q, cu_k, causal)
    ref = ref_np.varlen(q, k, v, cu_q, cu_k, causal)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


# --------------------------------------------------------------------------
# planted mistakes: each edit of the oracle source must fail a pin
# --------------------------------------------------------------------------

def _pins_hold(o) -> bool:
    """A compact run of the page-derived pins against oracle `o`."""
    try:
        # decode worked example: append slots
        g = load_golden("decode_block_table_example.txt")
        bs = g["block_size"]
        table = np.array([g["block_table_row0"], g["block_table_row1"], g["block_table_row2"]],
                         np.int32)
        rng = np.random.default_rng(0)
        kc = rng.standard_normal((8, bs, 2, 8)).astype(np.float32)
        vc = rng.standard_normal((8, bs, 2, 8)).astype(np.float32)
        kn = rng.standard_normal((3, 2, 8)).astype(np.float32)
        vn = rng.standard_normal((3, 2, 8)).astype(np.float32)
        o.decode(rng.standard_normal((3, 4, 8)).astype(np.float32), kc, vc, table,
                 np.array(g["cache_seqlens"], np.int32), kn, vn)
        for b in range(3):
            p, s = g["expected_append_block"][b], g["expected_append_slot"][b]
            if not np.array_equal(kc[p, s], kn[b]):
                return False
        # scalar-head example: exactly 3
        sh = load_golden("scalar_head_example.txt")
        kc = np.zeros((5, 4, 1, 1), np.float32)
        vc = np.zeros((5, 4, 1, 1), np.float32)
        for pos in range(4):
            vc[sh["placement_a"][pos // 4], pos % 4, 0, 0] = pos + 1
        out = o.decode(np.ones((1, 1, 1), np.float32), kc, vc,
                       np.array([sh["placement_a"]], np.int32), np.array([4], np.int32),
                       np.zeros((1, 1, 1), np.float32), np.full((1, 1, 1), 5.0, np.float32))
        if out[0, 0, 0] != 3.0:
            return False
        # GQA mapping (contiguous groups)
        hq, hkv, d = 4, 2, 2
        kc = rng.standard_normal((3, 4, hkv, d)).astype(np.float32)
        vc = np.zeros((3, 4, hkv, d), np.float32)
        vc[:, :, 1, :] = 1.0
        vn = np.zeros((1, hkv, d), np.float32)
        vn[0, 1] = 1.0
        out = o.decode(rng.standard_normal((1, hq, d)).astype(np.float32), kc, vc,
                       np.array([[0, 1, 2]], np.int32), np.array([9], np.int32),
                       rng.standard_normal((1, hkv, d)).astype(np.float32), vn)
        if not np.allclose(out[0, :, 0], [0, 0, 1, 1], atol=1e-14):
            return False
        # two-key closed form (scale)
        d = 16
        kc = np.zeros((2, 4, 1, d), np.float32)
        vc = np.zeros((2, 4, 1, d), np.float32)
        q = np.zeros((1, 1, d), np.float32)
        q[0, 0, 3] = 2.0
        kc[1, 0, 0, 3] = 1.5
        vc[1, 0, 0, :] = 1.0
        out = o.decode(q, kc, vc, np.array([[1, -1]], np.int32), np.array([1], np.int32),
                       np.zeros((1, 1, d), np.float32), np.full((1, 1, d), -2.0, np.float32))
        w = math.exp(3.0 / 4.0) / (math.exp(3.0 / 4.0) + 1.0)
        if not np.allclose(out[0, 0], w - 2.0 * (1 - w), rtol=1e-13):
            return False
        # causal bottom-right closed form
        ql, kl = 3, 8
        v = np.arange(kl, dtype=np.float32).reshape(kl, 1, 1)
        out = o.varlen(np.zeros((ql, 1, 1), np.float32), np.ones((kl, 1, 1), np.float32), v,
                       np.array([0, ql], np.int32), np.array([0, kl], np.int32), True)
        for i in range(ql):
            n = i + kl - ql + 1
            if not np.isclose(out[i, 0, 0], (n - 1) / 2, rtol=1e-13, atol=0):
                return False
        # cu_seq_lens example: empty key set for r0 gives zero rows
        cg = load_golden("cu_seq_lens_example.txt")
        q = rng.standard_normal((14, 1, 2)).astype(np.float32)
        k = rng.standard_normal((8, 1, 2)).astype(np.float32)
        out = o.varlen(q, k, k.copy(), np.array(cg["cu_seq_lens_q"], np.int32),
                       np.array(cg["cu_seq_lens_k"], np.int32), False)
        if not np.all(out[:10] == 0) or not np.array_equal(out[10, 0], k[0, 0].astype(float)):
            return False
        # cache update: chunk row i lands at logical position prefix + i
        kc = np.zeros((4, 4, 1, 1), np.float32)
        ch = np.array([1.0, 2.0, 3.0], np.float32).reshape(3, 1, 1)
        o.cache_update(ch, ch.copy(), np.array([0, 3], np.int32), np.array([2], np.int32),
                       np.array([[3, 0]], np.int32), kc, kc.copy())
        if not (kc[3, 2, 0, 0] == 1 and kc[3, 3, 0, 0] == 2 and kc[0, 0, 0, 0] == 3):
            return False
        return True
    except oracle.OracleError:
        return False


MUTATIONS = {
    "gqa interleaved": ("int hk = h / g;\n        int t = cache_seqlens[b] + 1;",
                        "int hk = h % num_kv_heads;\n        int t = cache_seqlens[b] + 1;"),
    "scale dropped": ("scores[j] = scale * dot;\n        }\n        /* passes 2 and 3",
                      "scores[j] = dot;\n        }\n        /* passes 2 and 3"),
    "new token not attended": ("int t = cache_seqlens[b] + 1;\n        double *scores",
                               "int t = cache_seqlens[b];\n        double *scores"),
    "append slot off by one": ("int rc = locate(block_table, b, cache_seqlens[b], block_size",
                               "int rc = locate(block_table, b, cache_seqlens[b] - 1, block_size"),
    "causal top-left": ("n = i + kl - ql + 1;", "n = i + 1;"),
    "weights not normalised": ("double w = exp(scores[j] - m) / l;", "double w = exp(scores[j] - m);"),
    "slot from block index": ("*slot = pos % block_size;", "*slot = pos / block_size;"),
    "values read from the key pool": ("softmax_weighted_sum(scores, t, v_cache, krow",
                                       "softmax_weighted_sum(scores, t, k_cache, krow"),
    "scatter ignores prefix": ("locate(block_table, b, prefix_lens[b] + i, block_size",
                               "locate(block_table, b, i, block_size"),
}


def test_unmodified_source_passes_pins(tmp_path):
    o = oracle.compile_variant(oracle.source_text(), str(tmp_path / "orig"))
    assert _pins_hold(o)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    src = oracle.source_text()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation anchor for {name!r} not unique"
    o = oracle.compile_variant(src.replace(old, new), str(tmp_path / name.replace(" ", "_")))
    assert not _pins_hold(o), f"planted mistake {name!r} slipped through the pins"

"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these expected values comes from the oracle itself or from the CUDA
path: they are the pages' worked examples (tests/golden/, each citing its
passage), closed forms, special cases and an independent numpy route.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import ref_np
from tests.conftest import bf16_bits, load_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _f32(*shape, seed=0, scale=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * scale).astype(np.float32)


# --------------------------------------------------------------------------
# decode worked example ("Perhatian berhalaman", Jalur decode / Contoh)
# --------------------------------------------------------------------------

def _worked_example_case(dtype=np.float32, seed=1):
    g = load_golden("decode_block_table_example.txt")
    bs = g["block_size"]
    table = np.array([g["block_table_row0"], g["block_table_row1"], g["block_table_row2"]],
                     dtype=np.int32)
    sl = np.array(g["cache_seqlens"], dtype=np.int32)
    hq, hkv, d, nb = 4, 2, 64, 8
    q = _f32(3, hq, d, seed=seed)
    kc = _f32(nb, bs, hkv, d, seed=seed + 1)
    vc = _f32(nb, bs, hkv, d, seed=seed + 2)
    kn = _f32(3, hkv, d, seed=seed + 3)
    vn = _f32(3, hkv, d, seed=seed + 4)
    if dtype == np.uint16:
        q, kc, vc, kn, vn = map(bf16_bits, (q, kc, vc, kn, vn))
    return g, q, kc, vc, table, sl, kn, vn


@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_decode_example_append_lands_where_the_page_says(dtype):
    g, q, kc, vc, table, sl, kn, vn = _worked_example_case(dtype)
    k0, v0 = kc.copy(), vc.copy()
    oracle.decode(q, kc, vc, table, sl, kn, vn)
    blocks, slots = g["expected_append_block"], g["expected_append_slot"]
    touched = np.zeros(kc.shape[:2], dtype=bool)
    for b in range(3):
        p, s = blocks[b], slots[b]
        assert np.array_equal(kc[p, s], kn[b]) and np.array_equal(vc[p, s], vn[b])
        touched[p, s] = True
    # every other slot of the pool is bit-for-bit unchanged
    assert np.array_equal(kc[~touched], k0[~touched])
    assert np.array_equal(vc[~touched], v0[~touched])


def test_decode_example_block_need():
    g = load_golden("decode_block_table_example.txt")
    bs = g["block_size"]
    rows = [g["block_table_row0"], g["block_table_row1"], g["block_table_row2"]]
    for L, row, need in zip(g["cache_seqlens"], rows, g["expected_blocks_needed_after_append"]):
        assert sum(1 for x in row if x >= 0) == need
        assert -(-(L + 1) // bs) == need  # the rule the example illustrates


def test_decode_example_output_uses_appended_token():
    """Attending over the 31/33/71 positions, with the new row included.

    The contiguous route is built by the test from the golden table, not by
    the oracle's own indexing."""
    g, q, kc, vc, table, sl, kn, vn = _worked_example_case()
    out = oracle.decode(q, kc.copy(), vc.copy(), table, sl, kn, vn)
    bs = g["block_size"]
    for b in range(3):
        L = g["cache_seqlens"][b]
        phys = [table[b][j // bs] for j in range(L)]
        krows = np.stack([kc[p, j % bs] for j, p in enumerate(phys)] + [kn[b]])
        vrows = np.stack([vc[p, j % bs] for j, p in enumerate(phys)] + [vn[b]])
        for h in range(4):
            ref = ref_np.attention(q[b, h][None].astype(np.float64),
                                   krows[:, h // 2].astype(np.float64),
                                   vrows[:, h // 2].astype(np.float64), 1 / 8.0)[0]
            np.testing.assert_allclose(out[b, h], ref, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# "39 · PagedAttention", 2. Phiên bản phân trang: the 60-token walk
# --------------------------------------------------------------------------

def test_block_walk_60_tokens():
    g = load_golden("block_walk_60_tokens.txt")
    bs, n = g["block_size"], g["length"]
    table = np.array([g["block_table"]], dtype=np.int32)
    nb = max(g["block_table"]) + 1
    d = 4
    rng = np.random.default_rng(5)
    # values: distinct random rows; keys: zero except one logical position
    vc = rng.standard_normal((nb, bs, 1, d)).astype(np.float32)
    kc = np.zeros((nb, bs, 1, d), dtype=np.float32)
    q = np.zeros((1, 1, d), dtype=np.float32)
    kn = np.zeros((1, 1, d), dtype=np.float32)
    vn = rng.standard_normal((1, 1, d)).astype(np.float32)
    # equal weights: output = mean of the values of exactly the walked slots
    walked = []
    for p, cnt in zip(g["expected_walk_physical"], g["expected_walk_tokens"]):
        walked += [(p, s) for s in range(cnt)]
    assert len(walked) == n
    out = oracle.decode(q, kc.copy(), vc.copy(), table, np.array([n - 1], np.int32), kn, vn)
    vals = [vc[p, s, 0] for p, s in walked[:-1]] + [vn[0, 0]]
    np.testing.assert_allclose(out[0, 0], np.mean(np.array(vals, np.float64), axis=0),
                               rtol=1e-12, atol=1e-14)
    # one dominant key at logical position 37 -> physical (12, 5) per the walk
    q[0, 0, 0] = 1.0
    kc[12, 5, 0, 0] = 400.0
    out = oracle.decode(q, kc.copy(), vc.copy(), table, np.array([n - 1], np.int32), kn, vn)
    np.testing.assert_allclose(out[0, 0], vc[12, 5, 0], rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# "PagedAttention" (paweldubiel.com): scalar head, output 3 in both placements
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
@pytest.mark.parametrize("placement", ["placement_a", "placement_b"])
def test_scalar_head_example(dtype, placement):
    g = load_golden("scalar_head_example.txt")
    bs, n = g["block_size"], g["positions"]
    phys = g[placement]
    nb = 5
    table = np.array([phys], dtype=np.int32)
    vals = np.array(g["values"], dtype=np.float32)
    kc = np.zeros((nb, bs, 1, 1), np.float32)
    vc = np.full((nb, bs, 1, 1), 99.0, np.float32)  # garbage elsewhere
    for pos in range(n - 1):
        vc[phys[pos // bs], pos % bs, 0, 0] = vals[pos]
    q = np.full((1, 1, 1), float(g["query"]), np.float32)
    kn = np.zeros((1, 1, 1), np.float32)
    vn = np.full((1, 1, 1), vals[n - 1], np.float32)
    if dtype == np.uint16:
        q, kc, vc, kn, vn = map(bf16_bits, (q, kc, vc, kn, vn))
    out = oracle.decode(q, kc, vc, table, np.array([n - 1], np.int32), kn, vn)
    assert out[0, 0, 0] == float(g["expected_output"])  # exactly 3


@pytest.mark.parametrize("placement", ["placement_a", "placement_b"])
def test_scalar_head_prefixes(placement):
    """Going from 1 to 5 positions (the 4 -> 5 step needs the second block)."""
    g = load_golden("scalar_head_example.txt")
    bs = g["block_size"]
    phys = g[placement]
    vals = np.array(g["values"], dtype=np.float32)
    for npos, want in zip(range(1, 6), g["expected_prefix_outputs"]):
        kc = np.zeros((5, bs, 1, 1), np.float32)
        vc = np.zeros((5, bs, 1, 1), np.float32)
        for pos in range(npos - 1):
            vc[phys[pos // bs], pos % bs, 0, 0] = vals[pos]
        used = -(-npos // bs)
        table = np.array([phys[:used] + [-1] * (2 - used)], dtype=np.int32)
        out = oracle.decode(np.ones((1, 1, 1), np.float32), kc, vc, table,
                            np.array([npos - 1], np.int32), np.zeros((1, 1, 1), np.float32),
                            np.full((1, 1, 1), vals[npos - 1], np.float32))
        assert out[0, 0, 0] == want


# --------------------------------------------------------------------------
# paged == contiguous ("not an approximation")
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_paged_equals_contiguous_bitwise(dtype):
    rng = np.random.default_rng(7)
    b, hq, hkv, d, bs, nb = 3, 4, 2, 16, 8, 40
    lens = np.array([0, 13, 57], np.int32)
    perm = rng.permutation(nb)
    table = np.full((b, 8), -1, np.int32)
    off = 0
    for i, L in enumerate(lens):
        n = -(-(L + 1) // bs)
        table[i, :n] = perm[off:off + n]
        off += n
    q, kc, vc = _f32(b, hq, d, seed=1), _f32(nb, bs, hkv, d, seed=2), _f32(nb, bs, hkv, d, seed=3)
    kn, vn = _f32(b, hkv, d, seed=4), _f32(b, hkv, d, seed=5)
    if dtype == np.uint16:
        q, kc, vc, kn, vn = map(bf16_bits, (q, kc, vc, kn, vn))
    out = oracle.decode(q, kc, vc, table, lens, kn, vn)  # kc/vc now hold the append
    for i, L in enumerate(lens):
        pos = np.arange(L + 1)
        kk = np.ascontiguousarray(kc[table[i, pos // bs], pos % bs])
        vv = np.ascontiguousarray(vc[table[i, pos // bs], pos % bs])
        for h in range(hq):
            ref = oracle.attend_contiguous(np.ascontiguousarray(q[i, h]), kk, vv, head=h // 2)
            assert np.array_equal(out[i, h], ref)


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------

def _one_seq(L, hq=2, hkv=1, d=8, bs=4, seed=0):
    rng = np.random.default_rng(seed)
    n = -(-(L + 1) // bs)
    nb = n + 3
    table = np.array([rng.permutation(nb)[:n]], np.int32)
    return table, nb, bs


def test_single_token_returns_new_value():
    table, nb, bs = _one_seq(0)
    kc, vc = _f32(nb, bs, 1, 8, seed=1), _f32(nb, bs, 1, 8, seed=2)
    vn = _f32(1, 1, 8, seed=3)
    out = oracle.decode(_f32(1, 2, 8, seed=4), kc, vc, table, np.array([0], np.int32),
                        _f32(1, 1, 8, seed=5), vn)
    assert np.array_equal(out[0, 0], vn[0, 0].astype(np.float64))
    assert np.array_equal(out[0, 1], vn[0, 0].astype(np.float64))


def test_equal_scores_give_mean_of_values():
    L = 22
    table, nb, bs = _one_seq(L)
    kc, vc = _f32(nb, bs, 1, 8, seed=1), _f32(nb, bs, 1, 8, seed=2)
    vn = _f32(1, 1, 8, seed=3)
    q = np.zeros((1, 2, 8), np.float32)
    out = oracle.decode(q, kc, vc, table, np.array([L], np.int32), _f32(1, 1, 8, seed=5), vn)
    pos = np.arange(L + 1)
    rows = vc[table[0, pos // bs], pos % bs, 0].astype(np.float64)
    np.testing.assert_allclose(out[0, 0], rows.mean(0), rtol=1e-13, atol=1e-15)


def test_two_key_softmax_closed_form_and_scale():
    """Scores a*s and 0 with s = 1/sqrt(D): weight e^(a s) / (e^(a s) + 1)."""
    d, bs = 16, 4
    table = np.array([[1, -1]], np.int32)
    kc = np.zeros((2, bs, 1, d), np.float32)
    vc = np.zeros((2, bs, 1, d), np.float32)
    q = np.zeros((1, 1, d), np.float32)
    q[0, 0, 3] = 2.0
    kc[1, 0, 0, 3] = 1.5          # q.k = 3.0 for position 0
    vc[1, 0, 0, :] = 1.0
    kn = np.zeros((1, 1, d), np.float32)  # q.k = 0 for the new token
    vn = np.full((1, 1, d), -2.0, np.float32)
    for scale_arg, s in ((0.0, 1 / math.sqrt(d)), (0.7, 0.7)):
        out = oracle.decode(q, kc.copy(), vc.copy(), table, np.array([1], np.int32), kn, vn,
                            softmax_scale=scale_arg)
        w = math.exp(3.0 * s) / (math.exp(3.0 * s) + 1.0)
        np.testing.assert_allclose(out[0, 0], w * 1.0 + (1 - w) * -2.0, rtol=1e-14)


@pytest.mark.parametrize("hq,hkv", [(4, 2), (8, 2), (8, 8), (6, 3)])
def test_gqa_head_mapping(hq, hkv):
    """q head h reads kv head h // (hq / hkv): contiguous groups."""
    L, d, bs = 9, 4, 4
    n = -(-(L + 1) // bs)
    table = np.array([list(range(n))], np.int32)
    kc = _f32(n, bs, hkv, d, seed=1)
    vc = np.zeros((n, bs, hkv, d), np.float32)
    for h in range(hkv):
        vc[:, :, h, :] = h + 1
    kn = _f32(1, hkv, d, seed=2)
    vn = np.arange(1, hkv + 1, dtype=np.float32).reshape(1, hkv, 1).repeat(d, 2)
    out = oracle.decode(_f32(1, hq, d, seed=3), kc, vc, table, np.array([L], np.int32), kn,
                        np.ascontiguousarray(vn))
    g = hq // hkv
    for h in range(hq):
        np.testing.assert_allclose(out[0, h], h // g + 1, rtol=1e-14)


def test_dominant_score_selects_its_value():
    L, d, bs = 30, 8, 8
    table, nb, bs = _one_seq(L, d=d, bs=bs, seed=3)
    kc = np.zeros((nb, bs, 1, d), np.float32)
    vc = _f32(nb, bs, 1, d, seed=4)
    q = np.zeros((1, 1, d), np.float32)
    q[0, 0, 0] = 1.0
    j = 17
    p, s = table[0, j // bs], j % bs
    kc[p, s, 0, 0] = 1000.0
    out = oracle.decode(q, kc, vc, table, np.array([L], np.int32), np.zeros((1, 1, d), np.float32),
                        _f32(1, 1, d, seed=6))
    np.testing.assert_allclose(out[0, 0], vc[p, s, 0], rtol=1e-14)


def test_unallocated_needed_block_is_an_error():
    table = np.array([[0, -1]], np.int32)
    kc = np.zeros((2, 4, 1, 2), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.decode(np.zeros((1, 1, 2), np.float32), kc, kc.copy(), table,
                      np.array([4], np.int32), np.zeros((1, 1, 2), np.float32),
                      np.zeros((1, 1, 2), np.float32))


# --------------------------------------------------------------------------
# varlen ("Perhatian berhalaman", Jalur Varlen / Contoh)
# --------------------------------------------------------------------------

def test_cu_seq_lens_example_indexing():
    g = load_golden("cu_seq_lens_example.txt")
    cu_q = np.array(g["cu_seq_lens_q"])
    cu_k = np.array(g["cu_seq_lens_k"])
    assert np.array_equal(np.diff(cu_q), g["q_lens"]) and np.array_equal(np.diff(cu_k), g["k_lens"])
    assert cu_q[-1] == g["total_q"] and cu_k[-1] == g["total_k"]
    assert max(g["q_lens"]) == g["max_length_q"] and max(g["k_lens"]) == g["max_length_k"]
    assert list(np.searchsorted(cu_q, np.arange(g["total_q"]), side="right") - 1) == g["q_request_index"]
    assert list(np.searchsorted(cu_k, np.arange(g["total_k"]), side="right") - 1) == g["k_request_index"]


@pytest.mark.parametrize("causal", [False, True])
def test_cu_seq_lens_example_outputs(causal):
    g = load_golden("cu_seq_lens_example.txt")
    cu_q = np.array(g["cu_seq_lens_q"], np.int32)
    cu_k = np.array(g["cu_seq_lens_k"], np.int32)
    hq, hkv, d = 4, 2, 8
    q = _f32(g["total_q"], hq, d, seed=1)
    k = _f32(g["total_k"], hkv, d, seed=2)
    v = _f32(g["total_k"], hkv, d, seed=3)
    out = oracle.varlen(q, k, v, cu_q, cu_k, causal)
    # r0 has no keys: its ten rows are zero
    assert np.array_equal(out[0:10], np.zeros((10, hq, d)))
    # r1 has one key (packed k row 0): a single key takes weight 1
    if causal:
        # ql=3, kl=1: query i sees key j iff j <= i - 2 -> only the last query
        assert np.array_equal(out[10:12], np.zeros((2, hq, d)))
        rows = [12]
    else:
        rows = [10, 11, 12]
    for r in rows:
        for h in range(hq):
            assert np.array_equal(out[r, h], v[0, h // 2].astype(np.float64))
    # r2: one query, seven keys; causal keeps all seven (j <= 0 + 7 - 1)
    ref = ref_np.attention(q[13, 0:1].astype(np.float64), k[1:8, 0].astype(np.float64),
                           v[1:8, 0].astype(np.float64), 1 / math.sqrt(d))
    np.testing.assert_allclose(out[13, 0], ref[0], rtol=1e-12)


@pytest.mark.parametrize("ql,kl", [(5, 5), (3, 8), (8, 3), (1, 1), (4, 0)])
def test_causal_alignment_closed_form(ql, kl):
    """q = 0: equal weights over the visible keys; value of key j = j.
    Bottom-right causal: query i sees n_i = clip(i + kl - ql + 1, 0, kl)
    keys, so the output is (n_i - 1) / 2, and 0 where n_i = 0."""
    d = 4
    q = np.zeros((ql, 1, d), np.float32)
    k = _f32(max(kl, 1), 1, d, seed=9)[:kl]
    v = np.arange(kl, dtype=np.float32).reshape(kl, 1, 1).repeat(d, 2)
    out = oracle.varlen(q, np.ascontiguousarray(k), np.ascontiguousarray(v),
                        np.array([0, ql], np.int32), np.array([0, kl], np.int32), True)
    for i in range(ql):
        n = min(max(i + kl - ql + 1, 0), kl)
        want = (n - 1) / 2 if n > 0 else 0.0
        np.testing.assert_allclose(out[i, 0], want, rtol=1e-14, atol=0)


# --------------------------------------------------------------------------
# cache update (scatter + gather)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_cache_update_scatter_and_gather(dtype):
    rng = np.random.default_rng(11)
    bs, hkv, d = 4, 2, 8
    q_lens = np.array([3, 0, 6, 1])
    prefix = np.array([5, 2, 0, 8])
    k_lens = q_lens + prefix
    need = -(-k_lens // bs)
    nb = int(need.sum()) + 4
    perm = rng.permutation(nb)
    table = np.full((4, int(need.max())), -1, np.int32)
    off = 0
    for i, n in enumerate(need):
        table[i, :n] = perm[off:off + n]
        off += n
    kc, vc = _f32(nb, bs, hkv, d, seed=1), _f32(nb, bs, hkv, d, seed=2)
    kch, vch = _f32(int(q_lens.sum()), hkv, d, seed=3), _f32(int(q_lens.sum()), hkv, d, seed=4)
    if dtype == np.uint16:
        kc, vc, kch, vch = map(bf16_bits, (kc, vc, kch, vch))
    cu_q = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(k_lens)]).astype(np.int32)
    k0, v0 = kc.copy(), vc.copy()
    kf, vf = oracle.cache_update(kch, vch, cu_q, prefix.astype(np.int32), table, kc, vc, cu_k)
    written = np.zeros((nb, bs), bool)
    for r in range(4):
        for i in range(q_lens[r]):
            pos = prefix[r] + i
            p, s = table[r, pos // bs], pos % bs
            assert np.array_equal(kc[p, s], kch[cu_q[r] + i])
            assert np.array_equal(vc[p, s], vch[cu_q[r] + i])
            written[p, s] = True
        # gather: prefix rows from the original pool, then the chunk rows
        for pos in range(k_lens[r]):
            src_k = (k0 if pos < prefix[r] else kc)[table[r, pos // bs], pos % bs]
            assert np.array_equal(kf[cu_k[r] + pos], src_k)
        np.testing.assert_array_equal(
            vf[cu_k[r]:cu_k[r + 1]], ref_np.gather_sequence(vc, table[r], int(k_lens[r]), bs))
    assert np.array_equal(kc[~written], k0[~written]) and np.array_equal(vc[~written], v0[~written])


def test_cache_update_rejects_inconsistent_cu_k():
    kc = np.zeros((4, 4, 1, 2), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.cache_update(np.zeros((2, 1, 2), np.float32), np.zeros((2, 1, 2), np.float32),
                            np.array([0, 2], np.int32), np.array([1], np.int32),
                            np.array([[0, 1]], np.int32), kc, kc.copy(),
                            np.array([0, 4], np.int32))


# --------------------------------------------------------------------------
# the (m, l) merge rule of "39 · PagedAttention", 3. Trên GPU
# --------------------------------------------------------------------------

def test_merge_rule_reproduces_one_softmax():
    rng = np.random.default_rng(3)
    s = rng.standard_normal(50) * 4
    v = rng.standard_normal((50, 6))
    w = np.exp(s - s.max())
    full = (w / w.sum()) @ v
    cuts = [0, 7, 7, 20, 49, 50]  # includes an empty part
    parts = [ref_np.partial(s[a:b], v[a:b]) for a, b in zip(cuts[:-1], cuts[1:])]
    acc = parts[0]
    for p in parts[1:]:
        acc = ref_np.merge_partials(acc, p)
    m, l, o = acc
    assert m == s.max()
    np.testing.assert_allclose(l, w.sum(), rtol=1e-13)
    np.testing.assert_allclose(o / l, full, rtol=1e-12, atol=1e-14)

"""Host-side checks of the seeded workload generators (no GPU)."""
import numpy as np
import pytest
import torch

from workloads import decode_config, make_decode, make_varlen, to_numpy, varlen_config
from tests.conftest import load_golden


def _check_tables(case, shared_ok=frozenset()):
    tab = case.block_table.numpy()
    bs = case.block_size
    seen = {}
    for b, L in enumerate(case.cache_seqlens.tolist()):
        n = -(-(L + 1) // bs)
        row = tab[b]
        assert (row[:n] >= 0).all() and (row[:n] < case.num_blocks).all()
        assert (row[n:] == -1).all()
        for p in row[:n]:
            if p in seen and p not in shared_ok:
                raise AssertionError(f"block {p} used by two sequences")
            seen[p] = b


def test_worked_example_config_is_the_pages_table():
    g = load_golden("decode_block_table_example.txt")
    c = decode_config(1)
    assert c.cache_seqlens.tolist() == g["cache_seqlens"]
    assert c.block_table.tolist() == [g["block_table_row0"], g["block_table_row1"],
                                      g["block_table_row2"]]
    assert c.q.dtype == torch.float32 and c.num_blocks == 8 and c.block_size == 32
    assert (c.num_heads, c.num_kv_heads, c.head_dim) == (4, 2, 64)


@pytest.mark.parametrize("idx", [2, 3])
def test_decode_configs_scaled(idx):
    c = decode_config(idx, scale_down=16)
    _check_tables(c)
    L = c.cache_seqlens.numpy()
    if idx == 2:
        assert L.min() >= 512 and L.max() <= 4096
    else:
        assert L.min() >= 64 and L.max() <= 32768


def test_shared_prefix_config_scaled():
    c = decode_config(5, scale_down=64)
    tab = c.block_table.numpy()
    shared = set(tab[0, :8].tolist())
    n_short = 1024 // 64
    for b in range(n_short):
        assert set(tab[b, :8].tolist()) == shared
        assert 257 <= c.cache_seqlens[b] <= 768
    _check_tables(c, shared_ok=frozenset(shared))
    # the append slot of every sequence is outside the shared blocks
    for b, L in enumerate(c.cache_seqlens.tolist()):
        assert tab[b, L // 32] not in shared
    assert c.unique_kv_bytes() < c.logical_kv_bytes()


def test_generators_are_deterministic():
    a = decode_config(2, scale_down=32)
    b = decode_config(2, scale_down=32)
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16))
    assert torch.equal(a.block_table, b.block_table)


def test_permutation_keeps_logical_content():
    c = decode_config(2, scale_down=32)
    p = c.permuted(7)
    bs = c.block_size
    for b, L in enumerate(c.cache_seqlens.tolist()[:3]):
        pos = np.arange(L + 1)
        a = to_numpy(c.k_cache)[c.block_table.numpy()[b, pos // bs], pos % bs]
        z = to_numpy(p.k_cache)[p.block_table.numpy()[b, pos // bs], pos % bs]
        assert np.array_equal(a, z)


def test_varlen_config_scaled():
    c = varlen_config(4, scale_down=16)
    cq, ck = c.cu_seq_lens_q.numpy(), c.cu_seq_lens_k.numpy()
    ql, kl = np.diff(cq), np.diff(ck)
    assert (kl == ql + c.prefix_lens.numpy()).all()
    assert c.max_length_q == ql.max() and c.max_length_k == kl.max()
    assert c.q.shape[0] == cq[-1] and c.k_chunk.shape[0] == cq[-1]
    tab = c.block_table.numpy()
    for r in range(c.batch):
        n = -(-int(kl[r]) // 16)
        assert (tab[r, :n] >= 0).all()


def test_causal_pair_count():
    c = make_varlen(1, [3, 5], [2, 0], 2, 1, 8, 4)
    # request 0: ql=3, kl=5 -> rows see 3, 4, 5 keys; request 1: 1..5
    assert c.causal_pairs() == 12 + 15

"""Host block manager: the pages' block-count rule, sharing with reference
counts, errors leave the state unchanged, and random-operation invariants."""
import numpy as np
import pytest

from paged_kv_cache_300_gb300 import _build
from tests.conftest import load_golden


@pytest.fixture(scope="module")
def BM():
    _build.build()
    from paged_kv_cache_300_gb300.blocks import BlockManager
    return BlockManager


def test_decode_example_block_counts(BM):
    """Docs page, decode example: 30, 32 and 70 cached tokens with blocks of
    32; after one new token each holds 1, 2 and 3 blocks."""
    g = load_golden("decode_block_table_example.txt")
    bm = BM(8, g["block_size"], g["max_blocks_per_seq"])
    for i, L in enumerate(g["cache_seqlens"]):
        bm.add(i, L)
    for i in range(3):
        bm.append(i, 1)
    table, lengths = bm.tables([0, 1, 2])
    held = (table >= 0).sum(1).tolist()
    assert held == g["expected_blocks_needed_after_append"]
    assert lengths.tolist() == [L + 1 for L in g["cache_seqlens"]]


def test_scalar_demo_fifth_token_needs_second_block(BM):
    """Blocks of 4: four tokens fit one block, the fifth takes a second and
    the first block (the prefix) does not move."""
    bm = BM(5, 4, 4)
    bm.add(7, 4)
    t0, _ = bm.tables([7])
    bm.append(7, 1)
    t1, _ = bm.tables([7])
    assert (t0 >= 0).sum() == 1 and (t1 >= 0).sum() == 2
    assert t1[0, 0] == t0[0, 0]


def test_shared_prefix_refcounts(BM):
    bm = BM(16, 4, 8)
    bm.add(1, 10)                       # 3 blocks, the last one partly full
    bm.fork(1, 2, 8)                    # shares the 2 full blocks
    bm.fork(1, 3, 8)
    t, L = bm.tables([1, 2, 3])
    shared = t[0, :2].tolist()
    assert t[1, :2].tolist() == shared and t[2, :2].tolist() == shared
    assert [bm.refcount(b) for b in shared] == [3, 3]
    assert L.tolist() == [10, 8, 8]
    bm.append(2, 1)                     # the child's next token: a block of its own
    t, _ = bm.tables([2])
    assert t[0, 2] not in shared and bm.refcount(int(t[0, 2])) == 1
    free_before = bm.num_free()
    bm.free(1)
    assert [bm.refcount(b) for b in shared] == [2, 2]
    assert bm.num_free() == free_before + 1  # only the parent's private block
    bm.free(2)
    bm.free(3)
    assert bm.num_free() == 16


def test_errors_leave_state_unchanged(BM):
    from paged_kv_cache_300_gb300.blocks import BlockManagerError
    bm = BM(4, 4, 3)
    bm.add(1, 8)
    with pytest.raises(BlockManagerError) as e:
        bm.add(2, 9)                     # needs 3 blocks, 2 free
    assert e.value.code == -4 and bm.num_free() == 2
    with pytest.raises(BlockManagerError) as e:
        bm.append(1, 5)                  # 13 tokens -> 4 blocks > max 3
    assert e.value.code == -5 and bm.length(1) == 8
    with pytest.raises(BlockManagerError):
        bm.fork(1, 3, 6)                 # not a multiple of the block size
    with pytest.raises(BlockManagerError):
        bm.add(1, 1)                     # id in use
    with pytest.raises(BlockManagerError):
        bm.free(9)
    assert bm.num_free() == 2 and bm.length(1) == 8


def test_random_operations_keep_invariants(BM):
    rng = np.random.default_rng(0)
    nb, bs, mb = 64, 4, 12
    bm = BM(nb, bs, mb)
    live = {}
    next_id = 0
    for _ in range(2000):
        op = rng.integers(0, 4)
        try:
            if op == 0 or not live:
                bm.add(next_id, int(rng.integers(0, 20)))
                live[next_id] = True
                next_id += 1
            elif op == 1:
                s = int(rng.choice(list(live)))
                bm.append(s, int(rng.integers(1, 6)))
            elif op == 2:
                s = int(rng.choice(list(live)))
                k = (bm.length(s) // bs) * bs
                bm.fork(s, next_id, int(rng.integers(0, k // bs + 1)) * bs)
                live[next_id] = True
                next_id += 1
            else:
                s = int(rng.choice(list(live)))
                bm.free(s)
                del live[s]
        except Exception as e:  # only capacity errors are expected
            assert getattr(e, "code", None) in (-4, -5), e
        ids = list(live)
        if not ids:
            continue
        t, L = bm.tables(ids)
        held = t[t >= 0].numpy()
        counts = np.bincount(held, minlength=nb)
        for b in range(nb):
            assert bm.refcount(b) == counts[b]
        assert bm.num_free() == int((counts == 0).sum())
        for row, n in zip(t.numpy(), L.numpy()):
            blocks = row[row >= 0]
            assert len(blocks) == -(-int(n) // bs)         # ceil(len / bs) blocks
            assert len(set(blocks.tolist())) == len(blocks)
            # a shared block is always full: the last block, if partly
            # filled, belongs to this sequence alone
            if n % bs and len(blocks):
                assert counts[blocks[-1]] == 1

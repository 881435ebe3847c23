"""GPU parity of pa_varlen_paged: keys read through the block table from the
pool.  Checked bit for bit against pa_cache_update (gather) + pa_varlen on the
same inputs, and within tolerance against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_300_gb300 as pa
from tests.gpu_util import assert_close, bits
from workloads import make_varlen, to_numpy, varlen_config

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pa.load()


def _both_paths(c, causal=True, err=None):
    """(fused output, gather + varlen output, gathered k, gathered v)."""
    t = lambda x: x.to("cuda")
    kc, vc = t(c.k_cache), t(c.v_cache)
    cq, ck, pl, bt = t(c.cu_seq_lens_q), t(c.cu_seq_lens_k), t(c.prefix_lens), t(c.block_table)
    q, kch, vch = t(c.q), t(c.k_chunk), t(c.v_chunk)
    tk = int(c.cu_seq_lens_k[-1])
    kf = torch.empty(tk, *c.k_chunk.shape[1:], dtype=c.k_chunk.dtype, device="cuda")
    vf = torch.empty_like(kf)
    pa.pa_cache_update(kch, vch, cq, pl, bt, kc, vc, kf, vf, ck)  # scatter + gather
    seqlens_k = (c.cu_seq_lens_k[1:] - c.cu_seq_lens_k[:-1]).to(torch.int32).cuda()
    fused = pa.pa_varlen_paged(q, kc, vc, bt, cq, seqlens_k, c.max_length_q, c.max_length_k,
                               causal, dev_err=err)
    ref = pa.pa_varlen(q, kf, vf, cq, ck, c.max_length_q, c.max_length_k, causal)
    torch.cuda.synchronize()
    return fused, ref, kf, vf


@pytest.mark.parametrize("bs", [8, 16, 32, 64])
@pytest.mark.parametrize("causal", [True, False])
def test_paged_equals_gather_path_bitwise(bs, causal):
    c = make_varlen(5 + bs, [1, 129, 300, 64, 255, 7, 0], [0, 17, 300, 5, 130, 513, 40], 8, 2,
                    128, bs, causal=causal)
    fused, ref, kf, vf = _both_paths(c, causal)
    assert torch.equal(fused.view(torch.int16), ref.view(torch.int16))
    o = oracle.varlen(to_numpy(c.q), bits(kf), bits(vf), c.cu_seq_lens_q.numpy(),
                      c.cu_seq_lens_k.numpy(), causal)
    assert_close(fused, o, torch.bfloat16, f"paged varlen bs={bs}")


def test_paged_workload_scaled_against_oracle():
    c = varlen_config(4, scale_down=8)
    fused, ref, kf, vf = _both_paths(c)
    assert torch.equal(fused.view(torch.int16), ref.view(torch.int16))
    o = oracle.varlen(to_numpy(c.q), bits(kf), bits(vf), c.cu_seq_lens_q.numpy(),
                      c.cu_seq_lens_k.numpy(), True)
    assert_close(fused, o, torch.bfloat16, "paged varlen, workload 4 scaled")


def test_paged_invariant_to_block_placement():
    c = make_varlen(9, [200, 70], [100, 300], 8, 2, 128, 16)
    g = torch.Generator().manual_seed(3)
    nb = c.k_cache.shape[0]
    pi = torch.randperm(nb, generator=g)
    inv = torch.empty_like(pi)
    inv[pi] = torch.arange(nb)
    c2 = make_varlen(9, [200, 70], [100, 300], 8, 2, 128, 16)
    c2.k_cache = c.k_cache[inv].clone()
    c2.v_cache = c.v_cache[inv].clone()
    m = c.block_table >= 0
    c2.block_table = c.block_table.clone()
    c2.block_table[m] = pi[c.block_table[m].long()].to(torch.int32)
    a, _, _, _ = _both_paths(c)
    b, _, _, _ = _both_paths(c2)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("bs,missing", [(16, 2), (16, 8), (8, 3), (8, 17), (64, 0), (64, 2)])
def test_paged_missing_block_flags_and_zeroes(bs, missing):
    """A needed -1 entry of request 0 (150 keys): a block of the first key
    tile, whose boxes go out before the block-wide barrier (bs=16 block 2,
    bs=8 block 3, bs=64 block 0), or of the third tile, loaded by the ring
    loop (bs=16 block 8, bs=8 block 17, bs=64 block 2).  Blocks of 8 and 16
    keys split a tile's boxes over three loader warps, blocks of 64 over
    two."""
    c = make_varlen(4, [50, 60], [100, 20], 8, 2, 128, bs)
    c.block_table[0, missing] = -1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t = lambda x: x.to("cuda")
    seqlens_k = (c.cu_seq_lens_k[1:] - c.cu_seq_lens_k[:-1]).to(torch.int32)
    out = pa.pa_varlen_paged(t(c.q), t(c.k_cache), t(c.v_cache), t(c.block_table),
                             t(c.cu_seq_lens_q), t(seqlens_k), c.max_length_q, c.max_length_k,
                             True, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEVERR_BAD_BLOCK
    assert torch.all(out[:50] == 0)
    assert not torch.all(out[50:] == 0)


def test_mixed_decode_and_prefill_in_one_launch():
    """A continuous-batching step: decode requests (one new token) and
    prefill chunks together, scattered with pa_cache_update and attended by
    one pa_varlen_paged launch.  Decode rows match pa_decode on the same
    state; every row matches the oracle."""
    q_lens = [1, 200, 1, 1, 57, 1]
    prefix = [300, 0, 17, 130, 400, 0]
    c = make_varlen(21, q_lens, prefix, 8, 2, 128, 16)
    t = lambda x: x.to("cuda")
    kc, vc = t(c.k_cache), t(c.v_cache)
    kc0, vc0 = kc.clone(), vc.clone()
    cq, bt, pl = t(c.cu_seq_lens_q), t(c.block_table), t(c.prefix_lens)
    q, kch, vch = t(c.q), t(c.k_chunk), t(c.v_chunk)
    pa.pa_cache_update(kch, vch, cq, pl, bt, kc, vc)
    seqlens_k = (c.cu_seq_lens_k[1:] - c.cu_seq_lens_k[:-1]).to(torch.int32).cuda()
    mixed = pa.pa_varlen_paged(q, kc, vc, bt, cq, seqlens_k, c.max_length_q, c.max_length_k, True)
    torch.cuda.synchronize()
    # the oracle on the gathered keys
    kf, vf = oracle.cache_update(to_numpy(c.k_chunk), to_numpy(c.v_chunk), c.cu_seq_lens_q.numpy(),
                                 c.prefix_lens.numpy(), c.block_table.numpy(),
                                 to_numpy(c.k_cache).copy(), to_numpy(c.v_cache).copy(),
                                 c.cu_seq_lens_k.numpy())
    ref = oracle.varlen(to_numpy(c.q), kf, vf, c.cu_seq_lens_q.numpy(), c.cu_seq_lens_k.numpy(),
                        True)
    assert_close(mixed, ref, torch.bfloat16, "mixed batch")
    # decode rows through the decode kernel on the pre-step pool
    dec = [r for r, n in enumerate(q_lens) if n == 1]
    rows = c.cu_seq_lens_q[dec].long()
    out_d = pa.pa_decode(q[rows.cuda()].contiguous(), kc0, vc0, bt[dec].contiguous(),
                         pl[dec].contiguous(), kch[rows.cuda()].contiguous(),
                         vch[rows.cuda()].contiguous())
    torch.cuda.synchronize()
    assert_close(out_d, mixed[rows.cuda()].double().cpu().numpy(), torch.bfloat16,
                 "decode kernel vs mixed launch")


def test_paged_long_request_past_the_staged_table():
    """bs=8 with 5000 keys: 625 table entries, more than the 512 the loaders
    stage in shared memory, so the rest are read from the table in global
    memory."""
    c = make_varlen(31, [100, 3], [4900, 700], 8, 2, 128, 8)
    assert c.block_table.shape[1] > 512
    fused, ref, kf, vf = _both_paths(c)
    assert torch.equal(fused.view(torch.int16), ref.view(torch.int16))
    o = oracle.varlen(to_numpy(c.q), bits(kf), bits(vf), c.cu_seq_lens_q.numpy(),
                      c.cu_seq_lens_k.numpy(), True)
    assert_close(fused, o, torch.bfloat16, "paged varlen, 5000 keys at bs=8")


@pytest.mark.parametrize("heads", [(4, 4), (8, 4), (16, 2)])
def test_paged_pack_factors(heads):
    """GQA groups of 1, 2 and 8 query heads through the block table."""
    hq, hkv = heads
    c = make_varlen(40 + hq, [3, 200, 65, 1], [40, 100, 0, 8], hq, hkv, 128, 16)
    fused, ref, kf, vf = _both_paths(c)
    assert torch.equal(fused.view(torch.int16), ref.view(torch.int16))
    o = oracle.varlen(to_numpy(c.q), bits(kf), bits(vf), c.cu_seq_lens_q.numpy(),
                      c.cu_seq_lens_k.numpy(), True)
    assert_close(fused, o, torch.bfloat16, f"paged varlen, {hq}/{hkv} heads")


@pytest.mark.parametrize("bs", [8, 16, 32, 64])
@pytest.mark.parametrize("causal", [True, False])
def test_paged_nan_in_unowned_pool_slots(bs, causal):
    """Every pool slot that holds no cached key (unused blocks, the tail of
    each request's last block, and the chunk slots before the scatter) holds
    NaN.  The keys past a request's length in its last block are read by the
    tile loads but weigh 0; the output must match the oracle (which reads
    only the request's keys), hold no NaN, and equal the gather path bit for
    bit."""
    c = make_varlen(50 + bs, [1, 129, 300, 64, 255, 7, 0, 33],
                    [0, 17, 300, 5, 130, 513, 40, 3], 8, 2, 128, bs, causal=causal)
    c.poison_unowned()
    fused, ref, kf, vf = _both_paths(c, causal)
    assert not torch.isnan(fused.float()).any()
    assert torch.equal(fused.view(torch.int16), ref.view(torch.int16))
    o = oracle.varlen(to_numpy(c.q), bits(kf), bits(vf), c.cu_seq_lens_q.numpy(),
                      c.cu_seq_lens_k.numpy(), causal)
    assert_close(fused, o, torch.bfloat16, f"NaN-poisoned pool, bs={bs} causal={causal}")


def test_mixed_batch_with_nan_in_unowned_pool_slots():
    """The continuous-batching step of test_mixed_decode_and_prefill_in_one_launch
    on a pool whose unwritten slots hold NaN."""
    q_lens = [1, 200, 1, 1, 57, 1]
    prefix = [300, 0, 17, 130, 400, 0]
    c = make_varlen(22, q_lens, prefix, 8, 2, 128, 16)
    c.poison_unowned()
    t = lambda x: x.to("cuda")
    kc, vc = t(c.k_cache), t(c.v_cache)
    cq, bt, pl = t(c.cu_seq_lens_q), t(c.block_table), t(c.prefix_lens)
    pa.pa_cache_update(t(c.k_chunk), t(c.v_chunk), cq, pl, bt, kc, vc)
    seqlens_k = (c.cu_seq_lens_k[1:] - c.cu_seq_lens_k[:-1]).to(torch.int32).cuda()
    mixed = pa.pa_varlen_paged(t(c.q), kc, vc, bt, cq, seqlens_k, c.max_length_q,
                               c.max_length_k, True)
    torch.cuda.synchronize()
    assert not torch.isnan(mixed.float()).any()
    kf, vf = oracle.cache_update(to_numpy(c.k_chunk), to_numpy(c.v_chunk), c.cu_seq_lens_q.numpy(),
                                 c.prefix_lens.numpy(), c.block_table.numpy(),
                                 to_numpy(c.k_cache).copy(), to_numpy(c.v_cache).copy(),
                                 c.cu_seq_lens_k.numpy())
    ref = oracle.varlen(to_numpy(c.q), kf, vf, c.cu_seq_lens_q.numpy(), c.cu_seq_lens_k.numpy(),
                        True)
    assert_close(mixed, ref, torch.bfloat16, "mixed batch, NaN-poisoned pool")


def test_varlen_packed_keys_next_request_nan():
    """Packed (gathered) keys: a request's last key tile reads the next
    request's rows; NaN there (a request whose own output is then NaN) must
    not reach the earlier request's output."""
    gen = torch.Generator().manual_seed(5)
    ql, kl = [40, 10], [70, 30]
    cu_q = torch.tensor([0, 40, 50], dtype=torch.int32)
    cu_k = torch.tensor([0, 70, 100], dtype=torch.int32)
    q = torch.randn(50, 8, 128, generator=gen).to(torch.bfloat16)
    k = torch.randn(100, 2, 128, generator=gen).to(torch.bfloat16)
    v = torch.randn(100, 2, 128, generator=gen).to(torch.bfloat16)
    k[70:], v[70:] = float("nan"), float("nan")
    out = pa.pa_varlen(q.cuda(), k.cuda(), v.cuda(), cu_q.cuda(), cu_k.cuda(), 40, 70, True)
    torch.cuda.synchronize()
    ref = oracle.varlen(to_numpy(q[:40]), to_numpy(k[:70]), to_numpy(v[:70]),
                        np.array([0, 40], np.int32), np.array([0, 70], np.int32), True)
    assert_close(out[:40], ref, torch.bfloat16, "request 0 next to a NaN request")

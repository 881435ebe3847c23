"""GPU parity of pa_cache_update (bit-exact) and pa_varlen (tolerance)
against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_300_gb300 as pa
from tests.conftest import load_golden
from tests.gpu_util import assert_close, bits
from workloads import make_varlen, to_numpy, varlen_config

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pa.load()


def _run_update(c, gather=True, dev="cuda"):
    t = lambda x: x.to(dev)
    kc, vc = t(c.k_cache), t(c.v_cache)
    kf = vf = ck = None
    if gather:
        tk = int(c.cu_seq_lens_k[-1])
        hkv, d = c.k_chunk.shape[1:]
        kf = torch.full((tk, hkv, d), float("nan"), dtype=c.k_chunk.dtype, device=dev)
        vf = torch.full_like(kf, float("nan"))
        ck = t(c.cu_seq_lens_k)
    pa.pa_cache_update(t(c.k_chunk), t(c.v_chunk), t(c.cu_seq_lens_q), t(c.prefix_lens),
                       t(c.block_table), kc, vc, kf, vf, ck)
    torch.cuda.synchronize()
    return kc, vc, kf, vf


def _oracle_update(c, gather=True):
    rk, rv = to_numpy(c.k_cache).copy(), to_numpy(c.v_cache).copy()
    kf, vf = oracle.cache_update(to_numpy(c.k_chunk), to_numpy(c.v_chunk),
                                 c.cu_seq_lens_q.numpy(), c.prefix_lens.numpy(),
                                 c.block_table.numpy(), rk, rv,
                                 c.cu_seq_lens_k.numpy() if gather else None)
    return rk, rv, kf, vf


@pytest.mark.parametrize("gather", [False, True])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_cache_update_bitwise(gather, dtype):
    c = make_varlen(3, [5, 0, 40, 16, 1], [11, 3, 0, 16, 200], 8, 2, 128, 16, dtype=dtype)
    kc, vc, kf, vf = _run_update(c, gather)
    rk, rv, rkf, rvf = _oracle_update(c, gather)
    assert np.array_equal(bits(kc), rk) and np.array_equal(bits(vc), rv)
    if gather:
        assert np.array_equal(bits(kf), rkf) and np.array_equal(bits(vf), rvf)


def test_cache_update_workload_scaled():
    c = varlen_config(4, scale_down=8)
    kc, vc, kf, vf = _run_update(c)
    rk, rv, rkf, rvf = _oracle_update(c)
    assert np.array_equal(bits(kc), rk) and np.array_equal(bits(vc), rv)
    assert np.array_equal(bits(kf), rkf) and np.array_equal(bits(vf), rvf)


def test_cache_update_bad_cu_k_flags():
    c = make_varlen(4, [5, 7], [3, 2], 8, 2, 64, 16)
    c.cu_seq_lens_k[2] += 1  # no longer prefix + q length
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t = lambda x: x.cuda()
    tk = int(c.cu_seq_lens_k[-1])
    kf = torch.zeros(tk, 2, 64, dtype=torch.bfloat16, device="cuda")
    pa.pa_cache_update(t(c.k_chunk), t(c.v_chunk), t(c.cu_seq_lens_q), t(c.prefix_lens),
                       t(c.block_table), t(c.k_cache), t(c.v_cache), kf, kf.clone(),
                       t(c.cu_seq_lens_k), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEVERR_BAD_CU


def _varlen_check(q, k, v, cu_q, cu_k, causal, dtype, max_q=None):
    dev = "cuda"
    ql = np.diff(cu_q.numpy())
    kl = np.diff(cu_k.numpy())
    if max_q is None:
        max_q = int(ql.max()) if len(ql) else 0
    out = pa.pa_varlen(q.to(dev), k.to(dev), v.to(dev), cu_q.to(dev), cu_k.to(dev),
                       max_q, int(kl.max()) if len(kl) else 0, causal)
    torch.cuda.synchronize()
    ref = oracle.varlen(to_numpy(q), to_numpy(k), to_numpy(v), cu_q.numpy(), cu_k.numpy(), causal)
    return out, ref, assert_close(out, ref, dtype, f"varlen causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_varlen_cu_seq_lens_example(causal, dtype):
    """The docs page's example: q lengths 10, 3, 1; k lengths 0, 1, 7."""
    g = load_golden("cu_seq_lens_example.txt")
    gen = torch.Generator().manual_seed(1)
    d = 128
    q = torch.randn(g["total_q"], 8, d, generator=gen).to(dtype)
    k = torch.randn(g["total_k"], 2, d, generator=gen).to(dtype)
    v = torch.randn(g["total_k"], 2, d, generator=gen).to(dtype)
    cu_q = torch.tensor(g["cu_seq_lens_q"], dtype=torch.int32)
    cu_k = torch.tensor(g["cu_seq_lens_k"], dtype=torch.int32)
    out, ref, _ = _varlen_check(q, k, v, cu_q, cu_k, causal, dtype)
    assert torch.all(out[:10].float() == 0)  # r0 has no keys


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_varlen_ragged_tiles(causal, dtype):
    """Lengths spanning several 128-row tiles with ragged tails, empty
    requests and ql > kl / ql < kl."""
    gen = torch.Generator().manual_seed(2)
    ql = [1, 129, 0, 300, 64, 255, 7]
    kl = [1, 400, 5, 300, 0, 130, 513]
    cu_q = torch.tensor([0] + list(np.cumsum(ql)), dtype=torch.int32)
    cu_k = torch.tensor([0] + list(np.cumsum(kl)), dtype=torch.int32)
    q = torch.randn(sum(ql), 8, 128, generator=gen).to(dtype)
    k = torch.randn(sum(kl), 2, 128, generator=gen).to(dtype)
    v = torch.randn(sum(kl), 2, 128, generator=gen).to(dtype)
    _varlen_check(q, k, v, cu_q, cu_k, causal, dtype)


@pytest.mark.parametrize("heads", [(4, 4), (8, 4), (16, 2)])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_pack_factors(heads, causal):
    """GQA groups of 1, 2 and 8 query heads: 1, 2 and 8 heads share each
    128-row tile."""
    hq, hkv = heads
    gen = torch.Generator().manual_seed(hq + hkv)
    ql = [3, 200, 65, 1, 130]
    kl = [40, 300, 65, 9, 129]
    cu_q = torch.tensor([0] + list(np.cumsum(ql)), dtype=torch.int32)
    cu_k = torch.tensor([0] + list(np.cumsum(kl)), dtype=torch.int32)
    q = torch.randn(sum(ql), hq, 128, generator=gen).to(torch.bfloat16)
    k = torch.randn(sum(kl), hkv, 128, generator=gen).to(torch.bfloat16)
    v = torch.randn(sum(kl), hkv, 128, generator=gen).to(torch.bfloat16)
    _varlen_check(q, k, v, cu_q, cu_k, causal, torch.bfloat16)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_many_items(causal):
    """Hundreds of short requests (some empty), a few long ones, and a
    max_length_q far above the longest request: many more work items than
    SMs, most of them empty, all taken over by the running CTAs."""
    gen = torch.Generator().manual_seed(11)
    rng = np.random.default_rng(11)
    n = 400
    ql = rng.integers(0, 6, n)
    ql[[7, 150, 399]] = [600, 257, 1000]
    kl = ql + rng.integers(0, 300, n)
    kl[[20, 21]] = 0
    ql[[20, 21]] = [0, 4]
    cu_q = torch.tensor([0] + list(np.cumsum(ql)), dtype=torch.int32)
    cu_k = torch.tensor([0] + list(np.cumsum(kl)), dtype=torch.int32)
    q = torch.randn(int(ql.sum()), 8, 128, generator=gen).to(torch.bfloat16)
    k = torch.randn(int(kl.sum()), 2, 128, generator=gen).to(torch.bfloat16)
    v = torch.randn(int(kl.sum()), 2, 128, generator=gen).to(torch.bfloat16)
    out, _, _ = _varlen_check(q, k, v, cu_q, cu_k, causal, torch.bfloat16, max_q=4000)
    assert torch.all(out[int(cu_q[21]):int(cu_q[22])] == 0)  # request 21 has no keys


def test_varlen_workload_scaled():
    """Workload 4 (scaled): scatter + gather, then causal varlen."""
    c = varlen_config(4, scale_down=8)
    kc, vc, kf, vf = _run_update(c)
    out, ref, _ = _varlen_check(c.q, kf.cpu(), vf.cpu(), c.cu_seq_lens_q, c.cu_seq_lens_k, True,
                                torch.bfloat16)


@pytest.mark.slow
def test_varlen_workload_full_sampled():
    """Full workload 4 in the benchmark's configuration; the oracle checks
    a sample of requests (varlen attention is independent per request)."""
    c = varlen_config(4)
    kc, vc, kf, vf = _run_update(c)
    rk, rv, rkf, rvf = _oracle_update(c)
    assert np.array_equal(bits(kf), rkf) and np.array_equal(bits(kc), rk)
    dev = "cuda"
    out = pa.pa_varlen(c.q.to(dev), kf, vf, c.cu_seq_lens_q.to(dev), c.cu_seq_lens_k.to(dev),
                       c.max_length_q, c.max_length_k, True)
    torch.cuda.synchronize()
    cq, ck = c.cu_seq_lens_q.numpy(), c.cu_seq_lens_k.numpy()
    for r in (0, int(np.argmax(np.diff(cq))), c.batch - 1):
        qs = to_numpy(c.q)[cq[r]:cq[r + 1]]
        ref = oracle.varlen(np.ascontiguousarray(qs), rkf[ck[r]:ck[r + 1]].copy(),
                            rvf[ck[r]:ck[r + 1]].copy(), np.array([0, len(qs)], np.int32),
                            np.array([0, ck[r + 1] - ck[r]], np.int32), True)
        assert_close(out[cq[r]:cq[r + 1]], ref, torch.bfloat16, f"request {r}")

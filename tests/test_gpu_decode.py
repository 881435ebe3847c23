"""GPU parity of pa_decode against the fp64 oracle (through the C ABI)."""
import math

import numpy as np
import pytest
import torch

import paged_kv_cache_300_gb300 as pa
from tests.conftest import load_golden
from tests.gpu_util import assert_close, bits, gpu_decode, oracle_decode, same_bits
from workloads import decode_config, make_decode, to_numpy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pa.load()


def _full_check(case, what):
    out, kc, vc = gpu_decode(case)
    ref, rk, rv = oracle_decode(case)
    assert same_bits(bits(kc), rk), f"{what}: K pool differs from the oracle's"
    assert same_bits(bits(vc), rv), f"{what}: V pool differs from the oracle's"
    return assert_close(out, ref, case.q.dtype, what)


def test_worked_example_fp32():
    """The decode example of the docs page, fp32, 1e-5; append slots bitwise."""
    case = decode_config(1)
    g = load_golden("decode_block_table_example.txt")
    out, kc, vc = gpu_decode(case)
    for b in range(3):
        p, s = g["expected_append_block"][b], g["expected_append_slot"][b]
        assert torch.equal(kc[p, s].cpu(), case.k_new[b]) and torch.equal(vc[p, s].cpu(), case.v_new[b])
    _full_check(case, "worked example")


@pytest.mark.parametrize("dtype,bs,npos,value", [(torch.float32, 4, 5, 3.0),
                                                 (torch.bfloat16, 16, 20, 10.5)])
@pytest.mark.parametrize("placement", ["placement_a", "placement_b"])
def test_scalar_head_example(dtype, bs, npos, value, placement):
    """Scalar-head example (paweldubiel.com) embedded in head_dim 64: keys 0,
    query e0, values 1..n in channel 0 -> exactly the mean, both placements.
    fp32 runs the page's block size 4; bf16 (block size 16 or 32) runs the
    same construction at block size 16 with 20 positions (mean 10.5)."""
    g = load_golden("scalar_head_example.txt")
    phys = g[placement]
    d = 64
    nb = 5
    kc = torch.zeros(nb, bs, 1, d, dtype=dtype)
    vc = torch.zeros(nb, bs, 1, d, dtype=dtype)
    vc[..., 1:] = 7.0  # other channels constant: output 7 there
    for pos in range(npos - 1):
        vc[phys[pos // bs], pos % bs, 0, 0] = pos + 1
    q = torch.zeros(1, 1, d, dtype=dtype)
    q[0, 0, 0] = 1.0
    vn = torch.zeros(1, 1, d, dtype=dtype)
    vn[..., 0] = npos
    vn[..., 1:] = 7.0
    tab = torch.tensor([phys], dtype=torch.int32)
    dev = "cuda"
    out = pa.pa_decode(q.to(dev), kc.to(dev), vc.to(dev), tab.to(dev),
                       torch.tensor([npos - 1], dtype=torch.int32, device=dev),
                       torch.zeros(1, 1, d, dtype=dtype, device=dev), vn.to(dev))
    o = out.float().cpu()[0, 0]
    assert o[0].item() == value
    assert torch.all(o[1:] == 7.0)
    if dtype == torch.float32:
        assert value == g["expected_output"]


@pytest.mark.parametrize("idx,scale", [(2, 16), (3, 32), (5, 128)])
def test_configs_scaled_down(idx, scale):
    case = decode_config(idx, scale_down=scale)
    _full_check(case, f"workload {idx} / {scale}")


@pytest.mark.parametrize("scale", [16, 4])
def test_workload2_shapes_unit_variance(scale):
    """Workload 2's exact shapes and launch path (GQA 32/8, head_dim 128,
    block size 16, L~U[512,4096], the 8-heads-per-CTA kernel) with N(0,1)
    values: outputs of order 0.1, so a wrong or zero output cannot pass
    under the absolute tolerance."""
    case = decode_config(2, scale_down=scale, unit_variance=True)
    _full_check(case, f"workload 2 N(0,1) / {scale}")
    out, _, _ = gpu_decode(case)
    assert float(out.float().abs().max()) > 0.05


@pytest.mark.parametrize("hq,hkv,d,bs,dtype", [(32, 8, 128, 16, torch.bfloat16),
                                               (8, 2, 64, 32, torch.bfloat16),
                                               (16, 4, 128, 32, torch.bfloat16),
                                               (32, 32, 64, 32, torch.bfloat16),
                                               (4, 2, 64, 16, torch.float32)])
def test_nan_in_unowned_pool_slots(hq, hkv, d, bs, dtype):
    """Every pool slot no sequence has written holds NaN (unused blocks, the
    tail of each last block, the append slot): what a pool allocated with
    uninitialised memory may hold.  The output must still match the oracle,
    which reads only the attended positions, and hold no NaN."""
    lens = [0, 1, bs - 1, bs, bs + 1, 3 * bs + 5, 700, 2000, 4 * bs - 2]
    case = make_decode(70 + d + bs, lens, hq, hkv, d, bs, dtype=dtype).poison_unowned()
    _full_check(case, f"NaN-poisoned pool hq={hq} hkv={hkv} d={d} bs={bs}")


@pytest.mark.parametrize("hq,hkv,d,bs", [(4, 4, 64, 16), (8, 4, 128, 16), (12, 4, 128, 32),
                                          (8, 1, 64, 32), (16, 2, 128, 16), (6, 2, 64, 16),
                                          (32, 4, 128, 32)])
def test_shapes_and_groups(hq, hkv, d, bs):
    rng = np.random.default_rng(hq * 100 + hkv * 10 + d + bs)
    lens = rng.integers(0, 700, size=7).tolist() + [0, bs - 1, bs, 2 * bs - 1]
    case = make_decode(7 + hq + d, lens, hq, hkv, d, bs)
    _full_check(case, f"hq={hq} hkv={hkv} d={d} bs={bs}")


def test_edge_lengths_single_token_and_block_boundaries():
    """L = 0 attends the new token only: out = v_new exactly (weight 1)."""
    case = make_decode(3, [0, 15, 16, 31, 32, 33], 8, 2, 128, 16)
    out, _, _ = gpu_decode(case)
    for h in range(8):
        assert torch.equal(out[0, h].cpu(), case.v_new[0, h // 4])
    _full_check(case, "edges")


def test_ragged_mix_many_splits():
    """Short and long sequences in one launch (stream-K split and merge)."""
    lens = [1, 5000, 17, 12000, 300, 0, 65, 9000]
    case = make_decode(11, lens, 16, 4, 128, 16)
    _full_check(case, "ragged mix")


def test_permutation_invariance_bitwise():
    case = decode_config(3, scale_down=32)
    perm = case.permuted(123)
    out_a, kc_a, vc_a = gpu_decode(case)
    out_b, kc_b, vc_b = gpu_decode(perm)
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    pi = perm.meta["perm"].cuda()
    assert torch.equal(kc_b[pi].view(torch.int16), kc_a.view(torch.int16))
    assert torch.equal(vc_b[pi].view(torch.int16), vc_a.view(torch.int16))


def test_repeatable_bitwise():
    case = decode_config(2, scale_down=8)
    a, _, _ = gpu_decode(case)
    b, _, _ = gpu_decode(case)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_bad_block_sets_error_and_zeroes_that_sequence():
    case = make_decode(5, [40, 100, 7], 8, 2, 64, 16)
    case.block_table[1, 3] = -1  # needed block of sequence 1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _, _ = gpu_decode(case, dev_err=err)
    assert int(err.item()) & pa.DEVERR_BAD_BLOCK
    assert torch.all(out[1] == 0)
    ref, _, _ = oracle_decode(case, rows=[0, 2])
    assert_close(out[[0, 2]], ref, torch.bfloat16, "good rows next to a bad one")


def test_length_overflow_sets_error():
    case = make_decode(6, [40, 30], 8, 2, 64, 16)
    case.cache_seqlens[1] = case.max_blocks_per_seq * 16  # no room for the new token
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _, _ = gpu_decode(case, dev_err=err)
    assert int(err.item()) & pa.DEVERR_OVERFLOW
    assert torch.all(out[1] == 0)


def test_host_side_misuse_returns_status():
    case = make_decode(1, [3], 8, 2, 96, 16)  # head_dim 96 unsupported
    with pytest.raises(pa.PAError) as e:
        gpu_decode(case)
    assert e.value.status == -4


@pytest.mark.slow
@pytest.mark.parametrize("idx,unit_variance", [(2, False), (2, True), (3, False), (5, False)])
def test_full_size_sampled(idx, unit_variance):
    """Full-size workload in the benchmark's launch configuration; the oracle
    checks a sample of sequences (the longest ones and a seeded draw), and
    the append of every sequence is checked bitwise.  Workload 2 also runs
    with N(0,1) values (same shapes), where its outputs are far above the
    absolute tolerance."""
    case = decode_config(idx, unit_variance=unit_variance)
    out, kc, vc = gpu_decode(case)
    L = case.cache_seqlens.numpy()
    rng = np.random.default_rng(idx)
    rows = sorted(set(np.argsort(L)[-2:].tolist() + rng.choice(len(L), 4, replace=False).tolist()))
    ref, _, _ = oracle_decode(case, rows=rows)
    assert_close(out[rows], ref, torch.bfloat16, f"workload {idx} sample {rows}")
    tab = case.block_table.numpy()
    kcb, knb = bits(kc), to_numpy(case.k_new)
    for b in range(len(L)):
        p, s = tab[b, L[b] // case.block_size], L[b] % case.block_size
        assert np.array_equal(kcb[p, s], knb[b])


def test_host_buffers_read_and_written_in_place():
    """q, block_table, cache_seqlens, k_new, v_new and out in page-locked host
    memory: the kernel reads and writes them in place (NVLink-C2C); the
    result equals the device-buffer call bit for bit, the append lands in
    the device pool, and the output matches the oracle."""
    case = decode_config(2, scale_down=8, unit_variance=True)
    dev_out, dev_k, dev_v = gpu_decode(case)
    kc, vc = case.k_cache.cuda(), case.v_cache.cuda()
    pin = lambda x: x.clone().pin_memory()
    host = [pin(x) for x in (case.q, case.block_table, case.cache_seqlens, case.k_new, case.v_new)]
    out = pa.pa_decode(host[0], kc, vc, host[1], host[2], host[3], host[4])
    torch.cuda.synchronize()
    assert not out.is_cuda and out.is_pinned()
    assert torch.equal(out.view(torch.int16), dev_out.cpu().view(torch.int16))
    assert torch.equal(kc.view(torch.int16), dev_k.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), dev_v.view(torch.int16))
    ref, _, _ = oracle_decode(case)
    assert_close(out, ref, torch.bfloat16, "host buffers")


def test_unpinned_host_tensors_are_refused():
    case = make_decode(2, [10, 20], 8, 2, 64, 16)
    with pytest.raises(ValueError):
        pa.pa_decode(case.q, case.k_cache.cuda(), case.v_cache.cuda(), case.block_table.cuda(),
                     case.cache_seqlens.cuda(), case.k_new.cuda(), case.v_new.cuda())

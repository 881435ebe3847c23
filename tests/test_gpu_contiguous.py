"""GPU parity of pa_decode_contiguous, the contiguous-cache twin of pa_decode
("39 · PagedAttention", inference-notes, sections "Ghi chú" and "4. Có miễn
phí không?": a paged kernel compared with one over a contiguous cache).

The contiguous cache [B, max_seqlen, Hkv, D] is filled here with the same
logical keys and values a paged case holds, so both calls see the same
attention problem: the twin must match pa_decode bit for bit (same kernel
code and split, only the address of a unit's rows differs), match the fp64
oracle's contiguous attention, and write the appended token in place.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_300_gb300 as pa
from tests.gpu_util import assert_close, bits, gpu_decode
from workloads import decode_config, make_decode, to_numpy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pa.load()


def contiguous_cache(case, max_seqlen=None, fill=float("nan")):
    return case.contiguous_cache(max_seqlen, fill, device="cuda")


def run_contiguous(case, kc, vc, dev_err=None):
    t = lambda x: x.to("cuda").contiguous()
    out = pa.pa_decode_contiguous(t(case.q), kc, vc, t(case.cache_seqlens), t(case.k_new),
                                  t(case.v_new), dev_err=dev_err)
    torch.cuda.synchronize()
    return out


def oracle_contiguous(case, kc, vc):
    """fp64 oracle over the contiguous rows, the append applied on the host
    copies first (position L of row b = the new token)."""
    k, v = bits(kc).copy(), bits(vc).copy()
    q, kn, vn = to_numpy(case.q), to_numpy(case.k_new), to_numpy(case.v_new)
    G = case.num_heads // case.num_kv_heads
    out = np.zeros(case.q.shape, dtype=np.float64)
    for b, L in enumerate(case.cache_seqlens.tolist()):
        k[b, L], v[b, L] = kn[b], vn[b]
        kr, vr = np.ascontiguousarray(k[b, :L + 1]), np.ascontiguousarray(v[b, :L + 1])
        for h in range(case.num_heads):
            out[b, h] = oracle.attend_contiguous(np.ascontiguousarray(q[b, h]), kr, vr, h // G)
    return out, k, v


@pytest.mark.parametrize("idx,scale,unit_variance", [(2, 16, True), (2, 8, False), (3, 32, False),
                                                     (5, 128, False)])
def test_contiguous_equals_paged_bitwise(idx, scale, unit_variance):
    case = decode_config(idx, scale_down=scale, unit_variance=unit_variance)
    kc, vc = contiguous_cache(case)
    out_c = run_contiguous(case, kc, vc)
    out_p, _, _ = gpu_decode(case)
    assert torch.equal(out_c.view(torch.int16), out_p.view(torch.int16))
    L = case.cache_seqlens.long()
    b = torch.arange(case.batch)
    assert torch.equal(kc[b, L].cpu(), case.k_new) and torch.equal(vc[b, L].cpu(), case.v_new)


@pytest.mark.parametrize("hq,hkv,d", [(8, 2, 128), (16, 4, 64), (4, 4, 64), (12, 4, 128)])
def test_contiguous_against_oracle(hq, hkv, d):
    lens = [0, 1, 15, 16, 17, 31, 32, 33, 300, 1000]
    case = make_decode(90 + hq + d, lens, hq, hkv, d, 16, value_scale=1.0)
    kc, vc = contiguous_cache(case, max_seqlen=1000 + 40)
    ref, rk, rv = oracle_contiguous(case, kc, vc)
    out = run_contiguous(case, kc, vc)
    assert_close(out, ref, torch.bfloat16, f"contiguous hq={hq} hkv={hkv} d={d}")
    # the append wrote position L of each row and nothing else
    assert np.array_equal(bits(kc), rk) and np.array_equal(bits(vc), rv)


def test_contiguous_row_end_not_multiple_of_unit():
    """max_seqlen not a multiple of the 16-token unit: a sequence's last unit
    reaches into the next row (or past the tensor); those rows weigh 0."""
    lens = [44, 12, 0, 44]
    case = make_decode(5, lens, 8, 2, 128, 16)
    kc, vc = contiguous_cache(case, max_seqlen=45)
    ref, _, _ = oracle_contiguous(case, kc, vc)
    out = run_contiguous(case, kc, vc)
    assert not torch.isnan(out.float()).any()
    assert_close(out, ref, torch.bfloat16, "max_seqlen 45")


def test_contiguous_overflow_flags_and_zeroes():
    case = make_decode(6, [40, 30, 10], 8, 2, 64, 16)
    kc, vc = contiguous_cache(case, max_seqlen=41)
    case.cache_seqlens[1] = 41  # no room for the new token
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_contiguous(case, kc, vc, dev_err=err)
    assert int(err.item()) & pa.DEVERR_OVERFLOW
    assert torch.all(out[1] == 0)
    assert not torch.all(out[0] == 0)


def test_contiguous_rejects_misuse():
    case = make_decode(7, [3], 8, 2, 96, 16)  # head_dim 96
    kc = torch.zeros(1, 8, 2, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pa.PAError) as e:
        run_contiguous(case, kc, kc.clone())
    assert e.value.status == -4

"""pa_decode_static_scratch: decode without a caller-supplied workspace.

Some callers cannot allocate device memory when they run a decode step (a
serving runtime with a fixed memory budget and no allocator in reach, a
plugin that is handed only its input and output buffers).  For them the
library keeps its split-K scratch in a fixed 16 MiB array of its own.  These
tests call that entry point through the C ABI and check it against the
regular pa_decode (which takes a workspace), bit for bit, on consecutive
calls of different shapes, and check that sizes beyond the array are
refused.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_300_gb300 as pa
from tests.gpu_util import bits
from workloads import decode_config

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pa.load()


def _run(fn, case):
    t = lambda x: x.to("cuda")
    kc, vc = t(case.k_cache), t(case.v_cache)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = fn(t(case.q), kc, vc, t(case.block_table), t(case.cache_seqlens), t(case.k_new),
             t(case.v_new), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out, kc, vc


def test_static_scratch_matches_pa_decode_on_consecutive_calls():
    # different shapes back to back: the shared array keeps the previous
    # call's contents, which must not leak into the next result
    cases = [decode_config(2, scale_down=8), decode_config(5, scale_down=128),
             decode_config(2, scale_down=8)]
    for n, case in enumerate(cases):
        ref_out, ref_k, ref_v = _run(pa.pa_decode, case)
        out, kc, vc = _run(pa.pa_decode_static_scratch, case)
        # same kernel, same plan, same merge order: equal bit for bit, so a
        # partial or counter left over from the previous call would show
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), f"call {n}"
        assert np.array_equal(bits(kc), bits(ref_k)) and np.array_equal(bits(vc), bits(ref_v))


def test_static_scratch_refuses_sizes_beyond_its_array():
    lib = pa.load()
    buf = torch.zeros(1024, dtype=torch.bfloat16, device="cuda")
    p = ctypes.c_void_p(buf.data_ptr())
    # 4096 sequences x 64 q heads x head_dim 128 need far more than 16 MiB
    need = pa.pa_decode_workspace_size(4096, 64, 8, 128, 16)
    assert need > (16 << 20)
    rc = lib.pa_decode_static_scratch(p, p, p, p, p, p, p, p, 4096, 64, 8, 128, 8, 16, 4, 0.0,
                                      None, None)
    assert rc == -5  # PA_ERR_WORKSPACE, nothing launched

"""The C ABI library loads and exports what include/pa.h declares; host-side
argument checks answer with status codes (no GPU needed: every case here is
rejected before the library touches CUDA)."""
import ctypes
import os
import re
import shutil

import pytest

import paged_kv_cache_300_gb300 as pa
from paged_kv_cache_300_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_build.LIB) and shutil.which("nvcc") is None and not os.path.exists(
            "/usr/local/cuda/bin/nvcc"):
        pytest.skip("library not built and no nvcc")
    _build.build()
    return pa.load()


def declared_functions():
    with open(os.path.join(ROOT, "include", "pa.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(pa_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("pa_decode", "pa_cache_update", "pa_varlen", "pa_decode_workspace_size",
              "pa_status_string", "pa_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/pa.h but not exported"


def test_status_strings_and_version(lib):
    assert pa.pa_status_string(0) == "ok"
    for code in range(-1, -8, -1):
        assert pa.pa_status_string(code) != "unknown status"
    assert pa.pa_version() >= 100


def _decode_args(**over):
    a = dict(q=1, k=1, v=1, bt=1, sl=1, kn=1, vn=1, out=1, batch=1, hq=8, hkv=2, d=64, nb=4, bs=16,
             mb=2, dtype=1, scale=0.0, ws=None, wsb=0, err=None, stream=None)
    a.update(over)
    p = lambda x: None if x is None else ctypes.c_void_p(x * 4096)
    return (p(a["q"]), p(a["k"]), p(a["v"]), p(a["bt"]), p(a["sl"]), p(a["kn"]), p(a["vn"]),
            p(a["out"]), a["batch"], a["hq"], a["hkv"], a["d"], a["nb"], a["bs"], a["mb"],
            a["dtype"], a["scale"], p(a["ws"]), a["wsb"], p(a["err"]), p(a["stream"]))


@pytest.mark.parametrize("over,status", [
    (dict(dtype=7), -2),
    (dict(hq=6, hkv=4), -3),
    (dict(batch=-1), -3),
    (dict(d=96), -4),
    (dict(q=None), -1),
    (dict(out=None), -1),
])
def test_decode_rejects_misuse_before_any_launch(lib, over, status):
    assert lib.pa_decode(*_decode_args(**over)) == status


def test_decode_empty_batch_is_a_no_op(lib):
    assert lib.pa_decode(*_decode_args(batch=0, q=None)) == 0


def test_varlen_and_cache_update_reject_misuse(lib):
    P = ctypes.c_void_p
    one = P(4096)
    # dtype
    assert lib.pa_varlen(one, one, one, one, one, 4, 4, 1, one, 1, 4, 4, 8, 2, 128, 9, 0.0, None,
                         None) == -2
    # unsupported head_dim
    assert lib.pa_varlen(one, one, one, one, one, 4, 4, 1, one, 1, 4, 4, 8, 2, 80, 1, 0.0, None,
                         None) == -4
    # group mismatch
    assert lib.pa_varlen(one, one, one, one, one, 4, 4, 1, one, 1, 4, 4, 6, 4, 128, 1, 0.0, None,
                         None) == -3
    # cache update: gather requested with a missing pointer
    assert lib.pa_cache_update(one, one, one, one, one, one, one, one, None, one, 1, 4, 4, 2, 128,
                               8, 16, 4, 1, None, None) == -1


def test_binding_refuses_cpu_tensors():
    import torch
    t = torch.zeros(1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pa.pa_decode(t, t, t, t, t, t, t)


def test_contiguous_decode_rejects_misuse_before_any_launch(lib):
    P = ctypes.c_void_p
    one = P(4096)

    def call(q=one, sl=one, batch=1, hq=8, hkv=2, d=128, lmax=64, ws=None):
        return lib.pa_decode_contiguous(q, one, one, sl, one, one, one, batch, hq, hkv, d, lmax,
                                        0.0, ws, 0, None, None)
    assert call(batch=0, q=None) == 0           # empty batch: nothing to do
    assert call(q=None) == -1                   # PA_ERR_NULL
    assert call(sl=None) == -1
    assert call(d=96) == -4                     # PA_ERR_UNSUPPORTED
    assert call(hq=6, hkv=4) == -3              # PA_ERR_SHAPE
    assert call(lmax=0) == -3
    assert call(q=P(4096 + 8)) == -3            # q not 16-byte aligned


def test_static_scratch_checks_pointers_before_touching_its_counters(lib):
    """A call refused for a null or misaligned pointer returns before it
    looks up or clears the library's scratch (no CUDA call at all: this
    machine may have no GPU)."""
    P = ctypes.c_void_p
    one = P(4096)
    rc = lib.pa_decode_static_scratch(one, one, one, one, one, one, one, None, 1, 8, 2, 128, 8,
                                      16, 4, 0.0, None, None)
    assert rc == -1
    rc = lib.pa_decode_static_scratch(P(4096 + 4), one, one, one, one, one, one, one, 1, 8, 2, 128,
                                      8, 16, 4, 0.0, None, None)
    assert rc == -3

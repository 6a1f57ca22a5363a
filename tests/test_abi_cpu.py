"""Host-side checks of the C ABI that need no GPU: the library loads, exports every symbol
include/sparse_mla.h declares, and rejects bad arguments with the documented status codes
before touching the device."""
import ctypes
import os
import re

import pytest

import sparse_mla_attention_fwd_gb300 as smla
from sparse_mla_attention_fwd_gb300 import _native
from sparse_mla_attention_fwd_gb300.native_build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sparse_mla.h")


@pytest.fixture(scope="module")
def lib():
    build()  # no-op when up to date; nvcc cross-compiles without a GPU
    return _native.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:smla_status|const char\*|int)\s+(sparse_mla_\w+)\s*\(", text, re.M)))


def test_header_declares_the_expected_entry_points():
    assert declared_functions() == sorted(_native.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_abi_version_and_status_strings(lib):
    assert lib.sparse_mla_abi_version() == 1
    for code in range(7):
        s = smla.sparse_mla_status_string(code)
        assert s and s != "unknown status"
    assert smla.sparse_mla_status_string(99) == "unknown status"


FAKE = 1 << 20  # 16-byte aligned non-null "device" address; never dereferenced on error paths


def call_fwd(lib, q=FAKE, kv=FAKE, idx=FAKE, tl=None, sink=None, scale=0.04, d_v=512, out=FAKE,
             lse=FAKE, mx=FAKE, s_q=4, s_kv=16, h_q=64, d_qk=512, topk=8):
    return lib.sparse_mla_fwd(q, kv, idx, tl, sink, ctypes.c_float(scale), d_v, out, lse, mx, s_q,
                              s_kv, h_q, d_qk, topk, None)


@pytest.mark.parametrize("kw,code", [
    (dict(h_q=48), 2), (dict(h_q=0), 2), (dict(d_qk=256), 2), (dict(d_v=256), 2),
    (dict(topk=0), 2), (dict(s_q=-1), 2), (dict(scale=0.0), 2), (dict(scale=float("nan")), 2),
    (dict(s_kv=-3), 2), (dict(q=None), 1), (dict(idx=None), 1), (dict(out=None), 1),
    (dict(lse=None), 1), (dict(mx=None), 1), (dict(q=FAKE + 4), 3), (dict(kv=FAKE + 8), 3),
    (dict(idx=FAKE + 2), 3), (dict(s_q=1 << 26, h_q=128), 2),
])
def test_bad_arguments_are_rejected_without_launch(lib, kw, code):
    assert call_fwd(lib, **kw) == code


def test_zero_rows_is_ok_without_a_device(lib):
    assert call_fwd(lib, s_q=0, q=None, kv=None, idx=None, out=None, lse=None, mx=None) == 0


def test_paged_argument_checks(lib):
    f = lib.sparse_mla_fwd_paged
    base = dict(q=FAKE, pool=FAKE, rows=4096, bt=FAKE, max_blocks=64, page=64, seqlens=None,
                s_kv=4096, sq_req=1, idx=FAKE, tl=None, sink=None, scale=0.04, d_v=512, out=FAKE,
                lse=FAKE, mx=FAKE, s_q=8, h_q=128, d_qk=576, topk=2048)

    def call(**kw):
        a = dict(base, **kw)
        return f(a["q"], a["pool"], a["rows"], a["bt"], a["max_blocks"], a["page"], a["seqlens"],
                 a["s_kv"], a["sq_req"], a["idx"], a["tl"], a["sink"], ctypes.c_float(a["scale"]),
                 a["d_v"], a["out"], a["lse"], a["mx"], a["s_q"], a["h_q"], a["d_qk"], a["topk"], None)

    assert call(bt=None) == 1
    assert call(page=0) == 2
    assert call(max_blocks=0) == 2
    assert call(rows=0) == 2
    assert call(sq_req=3) == 2  # s_q not a multiple of s_q_per_req
    assert call(bt=FAKE + 2) == 3
    assert call(s_q=0, q=None) == 0


def test_python_wrapper_rejects_cpu_tensors():
    import torch
    q = torch.zeros((2, 64, 512), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        smla.sparse_mla_fwd(q, q, torch.zeros((2, 1, 4), dtype=torch.int32))

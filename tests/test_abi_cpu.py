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
    return sorted(set(re.findall(r"^\s*(?:smla_status|const char\*|int|size_t)\s+(sparse_mla_\w+)\s*\(", text, re.M)))


def test_header_declares_the_expected_entry_points():
    assert declared_functions() == sorted(_native.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_abi_version_and_status_strings(lib):
    assert lib.sparse_mla_abi_version() == 4
    for code in range(8):
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


def test_splitkv_workspace_size_and_argument_checks(lib):
    size = lib.sparse_mla_splitkv_workspace_size
    assert size(4, 64, 1) == 0                      # one range needs no workspace
    units = 4 * 2 * 3
    o_bytes = units * 64 * 512 * 4
    assert size(4, 128, 3) == ((o_bytes + 255) // 256) * 256 + units * 3 * 64 * 4
    assert size(4, 64, 0) == 0 and size(4, 64, 65) == 0 and size(4, 48, 2) == 0
    f = lib.sparse_mla_fwd_splitkv

    def call(n_split=2, ws=FAKE, nbytes=1 << 30, **kw):
        a = dict(q=FAKE, kv=FAKE, idx=FAKE, out=FAKE, s_q=4, h_q=64, topk=256)
        a.update(kw)
        return f(a["q"], a["kv"], a["idx"], None, None, ctypes.c_float(0.04), 512, a["out"], FAKE, FAKE,
                 a["s_q"], 1000, a["h_q"], 512, a["topk"], n_split, ws, nbytes, None)

    assert call(n_split=0) == 2 and call(n_split=65) == 2
    assert call(ws=None) == 7                       # missing workspace
    assert call(nbytes=1000) == 7                   # too small
    assert call(ws=FAKE + 16) == 3                  # not 256-byte aligned
    assert call(s_q=0, q=None, kv=None, idx=None, out=None) == 0
    assert call(s_q=0, ws=None) == 0                # no rows: the workspace is not inspected


def call_bwd(lib, q=FAKE, kv=FAKE, out=FAKE, dout=FAKE, idx=FAKE, tl=None, sink=None, lse=FAKE, scale=0.04,
             d_v=512, dq=FAKE, dkv=FAKE, dsink=None, s_q=4, s_kv=16, h_q=64, d_qk=576, topk=8):
    return lib.sparse_mla_bwd(q, kv, out, dout, idx, tl, sink, lse, ctypes.c_float(scale), d_v, dq, dkv, dsink,
                              s_q, s_kv, h_q, d_qk, topk, None)


@pytest.mark.parametrize("kw,code", [
    (dict(h_q=48), 2), (dict(d_qk=256), 2), (dict(d_v=256), 2), (dict(topk=0), 2), (dict(s_kv=-1), 2),
    (dict(scale=-1.0), 2), (dict(q=None), 1), (dict(idx=None), 1), (dict(lse=None), 1), (dict(dq=None), 1),
    (dict(out=None), 1), (dict(dout=None), 1), (dict(dkv=None), 1), (dict(out=FAKE + 8), 3),
    (dict(dout=FAKE + 4), 3), (dict(q=FAKE + 2), 3), (dict(dkv=FAKE + 2), 3), (dict(dsink=FAKE + 1), 3),
    (dict(sink=FAKE + 2), 3), (dict(tl=FAKE + 2), 3),
])
def test_bwd_rejects_bad_arguments_before_any_launch(lib, kw, code):
    assert call_bwd(lib, **kw) == code


def test_host_entry_rejects_bad_arguments_before_any_copy(lib):
    f = lib.sparse_mla_fwd_host

    def call(q_h=FAKE, kv_h=FAKE, idx_h=FAKE, tl_h=None, sink_h=None, out_h=FAKE, tl_d=None, sink_d=None,
             n_chunks=4, s_q=16, q_d=FAKE):
        return f(q_h, kv_h, idx_h, tl_h, sink_h, ctypes.c_float(0.04), 512, out_h, FAKE, FAKE, s_q, 100, 64, 576,
                 32, q_d, FAKE, FAKE, tl_d, sink_d, FAKE, FAKE, FAKE, n_chunks, None, None, None)

    assert call(n_chunks=0) == 2 and call(n_chunks=65) == 2
    assert call(q_h=None) == 1 and call(kv_h=None) == 1 and call(out_h=None) == 1
    assert call(tl_h=FAKE) == 1 and call(tl_d=FAKE) == 1          # host and device must match
    assert call(sink_h=FAKE) == 1
    assert call(q_d=FAKE + 8) == 3
    assert call(s_q=0, q_h=None, out_h=None) == 0                   # no rows: nothing is inspected

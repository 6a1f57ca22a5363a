"""CPU fp64 oracle for the sparse MLA attention forward (DSA top-k).

TEST INFRASTRUCTURE ONLY.  This package is the reference the CUDA path is checked against.
Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it; the product package never does, and it shares no code with the CUDA path.

The arithmetic lives in ``sparse_mla_oracle.c`` (plain C, IEEE double, no fast-math), which
states the definition it follows and cites the passages of the FlashMLA pull requests that fix
each part.  This module only builds that file with gcc and marshals numpy arrays into it.

Inputs are passed exactly as the GPU receives them: q / kv as bf16 bit patterns (uint16),
indices / topk_length as int32, attn_sink as float32, sm_scale as the float32 value.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sparse_mla_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libsmla_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, -O2, OpenMP).  Returns its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    P = ctypes.c_void_p
    I64, I32, D = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    lib.smla_oracle_fwd.restype = ctypes.c_int
    lib.smla_oracle_fwd.argtypes = [P, P, P, P, P, D, I64, I64, I32, I32, I32, I32, P, I64,
                                    P, P, P, I32]
    lib.smla_oracle_fwd_paged.restype = ctypes.c_int
    lib.smla_oracle_fwd_paged.argtypes = [P, P, P, P, I64, I32, I32, I32, P, P, P, D, I64,
                                          I32, I32, I32, I32, P, I64, P, P, P, I32]
    lib.smla_oracle_last_valid_length.restype = None
    lib.smla_oracle_last_valid_length.argtypes = [P, I64, I32, I64, P]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def sparse_mla_fwd(q_bits, kv_bits, indices, topk_length=None, attn_sink=None, sm_scale=None,
                   d_v=512, rows=None, threads=0, _lib_=None):
    """fp64 reference.  q_bits [s_q, h_q, d_qk] uint16, kv_bits [s_kv, 1, d_qk] (or [s_kv, d_qk])
    uint16, indices [s_q, 1, topk] (or [s_q, topk]) int32.  Returns (O, lse, max_logits) as
    float64 arrays of shape [n, h_q, d_v], [n, h_q], [n, h_q] for the listed rows (all rows when
    ``rows`` is None)."""
    lib = _lib_ or _load()
    q_bits = _c(q_bits, np.uint16)
    kv_bits = _c(kv_bits, np.uint16)
    indices = _c(indices, np.int32)
    s_q, h_q, d_qk = q_bits.shape
    s_kv = kv_bits.shape[0]
    topk = indices.reshape(s_q, -1).shape[1]
    if sm_scale is None:
        sm_scale = float(np.float32(1.0 / np.sqrt(d_qk)))
    rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = s_q if rows_arr is None else len(rows_arr)
    out = np.empty((n, h_q, d_v), np.float64)
    lse = np.empty((n, h_q), np.float64)
    mx = np.empty((n, h_q), np.float64)
    tl = _c(topk_length, np.int32)
    sink = _c(attn_sink, np.float32)
    rc = lib.smla_oracle_fwd(_ptr(q_bits), _ptr(kv_bits), _ptr(indices), _ptr(tl), _ptr(sink),
                             float(sm_scale), s_q, s_kv, h_q, d_qk, d_v, topk, _ptr(rows_arr), n,
                             _ptr(out), _ptr(lse), _ptr(mx), int(threads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments (bad row id or out of memory)")
    return out, lse, mx


def sparse_mla_fwd_paged(q_bits, kv_pool_bits, block_table, indices, page_block=64,
                         seqlens_k=None, s_kv_per_req=0, s_q_per_req=1, topk_length=None,
                         attn_sink=None, sm_scale=None, d_v=512, rows=None, threads=0, _lib_=None):
    """fp64 reference over a paged KV cache; same outputs as :func:`sparse_mla_fwd`."""
    lib = _lib_ or _load()
    q_bits = _c(q_bits, np.uint16)
    kv_pool_bits = _c(kv_pool_bits, np.uint16)
    block_table = _c(block_table, np.int32)
    indices = _c(indices, np.int32)
    s_q, h_q, d_qk = q_bits.shape
    topk = indices.reshape(s_q, -1).shape[1]
    max_blocks = block_table.shape[1]
    if sm_scale is None:
        sm_scale = float(np.float32(1.0 / np.sqrt(d_qk)))
    rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = s_q if rows_arr is None else len(rows_arr)
    out = np.empty((n, h_q, d_v), np.float64)
    lse = np.empty((n, h_q), np.float64)
    mx = np.empty((n, h_q), np.float64)
    sk = _c(seqlens_k, np.int32)
    tl = _c(topk_length, np.int32)
    sink = _c(attn_sink, np.float32)
    rc = lib.smla_oracle_fwd_paged(_ptr(q_bits), _ptr(kv_pool_bits), _ptr(block_table), _ptr(sk),
                                   int(s_kv_per_req), max_blocks, int(page_block), int(s_q_per_req),
                                   _ptr(indices), _ptr(tl), _ptr(sink), float(sm_scale), s_q, h_q,
                                   d_qk, d_v, topk, _ptr(rows_arr), n, _ptr(out), _ptr(lse),
                                   _ptr(mx), int(threads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out, lse, mx


def last_valid_length(indices, s_kv, _lib_=None):
    """One past the last slot holding 0 <= idx < s_kv in each row (0 for rows without one)."""
    lib = _lib_ or _load()
    indices = _c(indices, np.int32)
    s_q = indices.shape[0]
    topk = indices.reshape(s_q, -1).shape[1]
    out = np.empty(s_q, np.int32)
    lib.smla_oracle_last_valid_length(_ptr(indices), s_q, topk, int(s_kv), _ptr(out))
    return out


class Variant:
    """The same three calls bound to another build of the oracle source (a shared library at
    ``path``).  The pin tests use it to check that planted mistakes in the arithmetic are
    caught; nothing else does."""

    def __init__(self, path):
        self._lib = _bind(ctypes.CDLL(path))

    def sparse_mla_fwd(self, *a, **kw):
        return sparse_mla_fwd(*a, _lib_=self._lib, **kw)

    def sparse_mla_fwd_paged(self, *a, **kw):
        return sparse_mla_fwd_paged(*a, _lib_=self._lib, **kw)

    def last_valid_length(self, *a, **kw):
        return last_valid_length(*a, _lib_=self._lib, **kw)

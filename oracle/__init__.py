"""CPU fp64 oracle for the sparse MLA attention forward and backward (DSA top-k).

TEST INFRASTRUCTURE ONLY.  This package is the reference the CUDA path is checked against.
Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it; the product package never does, and it shares no code with the CUDA path.

The arithmetic lives in ``sparse_mla_oracle.c`` (forward) and ``sparse_mla_bwd_oracle.c``
(backward: the gradients of sum(dO * O)), plain C in IEEE double without fast-math; each states
the definition it follows and cites the passages of the FlashMLA pull requests that fix each
part.  This module only builds those files with gcc and marshals numpy arrays into them.

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
_BWD_SRC = os.path.join(_HERE, "sparse_mla_bwd_oracle.c")
_BWD_LIB_PATH = os.path.join(_BUILD_DIR, "libsmla_bwd_oracle.so")
_lock = threading.Lock()
_lib = None
_bwd_lib = None


def _compile(src, lib_path, force):
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(lib_path)) or os.path.getmtime(lib_path) < os.path.getmtime(src)
    if force or stale:
        tmp = lib_path + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-shared", "-fPIC", "-o", tmp, src, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib_path)
    return lib_path


def build(force: bool = False) -> str:
    """Compile the oracle shared libraries (gcc, -O2, OpenMP).  Returns the forward's path."""
    _compile(_BWD_SRC, _BWD_LIB_PATH, force)
    return _compile(_SRC, _LIB_PATH, force)


def _bind(lib):
    P = ctypes.c_void_p
    I64, I32, D = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    lib.smla_oracle_fwd.restype = ctypes.c_int
    lib.smla_oracle_fwd.argtypes = [P, P, P, P, P, D, I64, I64, I32, I32, I32, I32, P, I64,
                                    P, P, P, I32]
    lib.smla_oracle_fwd_paged.restype = ctypes.c_int
    lib.smla_oracle_fwd_paged.argtypes = [P, P, I64, P, P, I64, I32, I32, I32, P, P, P, D, I64,
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
    """fp64 reference over a paged KV cache [pool_rows, 1, d_qk] with a block table
    [n_req, max_blocks]; same outputs as :func:`sparse_mla_fwd`.  A position past the request's
    length or its table row, on a negative table entry, or on a row past the pool is an invalid
    slot."""
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
    pool_rows = kv_pool_bits.shape[0]
    rc = lib.smla_oracle_fwd_paged(_ptr(q_bits), _ptr(kv_pool_bits), pool_rows, _ptr(block_table), _ptr(sk),
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


# ---------------------------------------------------------------------------------- backward
def _bind_bwd(lib):
    P, I64, I32, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
    lib.smla_oracle_bwd.restype = ctypes.c_int
    lib.smla_oracle_bwd.argtypes = [P, P, P, P, P, P, D, I64, I64, I32, I32, I32, I32, P, P, P, I32]
    return lib


def _load_bwd():
    global _bwd_lib
    with _lock:
        if _bwd_lib is None:
            build()
            _bwd_lib = _bind_bwd(ctypes.CDLL(_BWD_LIB_PATH))
    return _bwd_lib


def bf16_bits_to_f64(bits):
    """bf16 bit patterns (uint16) -> float64, exactly."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def sparse_mla_bwd_f64(q, kv, dout, indices, topk_length=None, attn_sink=None, sm_scale=None,
                       threads=0, _lib_=None):
    """fp64 gradients of sum(dout * O) for real-valued inputs.  q [s_q, h_q, d_qk],
    kv [s_kv, d_qk] (or [s_kv, 1, d_qk]), dout [s_q, h_q, d_v] float64; indices [s_q, topk]
    (or [s_q, 1, topk]) int32.  Returns (dq [s_q, h_q, d_qk], dkv [s_kv, d_qk], dsink [h_q] or
    None) as float64."""
    lib = _lib_ or _load_bwd()
    q = np.ascontiguousarray(q, dtype=np.float64)
    dout = np.ascontiguousarray(dout, dtype=np.float64)
    s_q, h_q, d_qk = q.shape
    kv = np.ascontiguousarray(kv, dtype=np.float64).reshape(-1, d_qk)
    s_kv = kv.shape[0]
    d_v = dout.shape[2]
    indices = _c(indices, np.int32).reshape(s_q, -1)
    topk = indices.shape[1]
    if sm_scale is None:
        sm_scale = float(np.float32(1.0 / np.sqrt(d_qk)))
    dq = np.empty((s_q, h_q, d_qk), np.float64)
    dkv = np.empty((s_kv, d_qk), np.float64)
    sink = _c(attn_sink, np.float32)
    dsink = np.empty(h_q, np.float64) if sink is not None else None
    tl = _c(topk_length, np.int32)
    rc = lib.smla_oracle_bwd(_ptr(q), _ptr(kv), _ptr(dout), _ptr(indices), _ptr(tl), _ptr(sink),
                             float(sm_scale), s_q, s_kv, h_q, d_qk, d_v, topk, _ptr(dq), _ptr(dkv),
                             _ptr(dsink), int(threads))
    if rc != 0:
        raise ValueError("backward oracle ran out of memory")
    return dq, dkv, dsink


def sparse_mla_bwd(q_bits, kv_bits, dout_bits, indices, topk_length=None, attn_sink=None,
                   sm_scale=None, threads=0, _lib_=None):
    """fp64 gradients of sum(dout * O) for bf16 inputs given as bit patterns (uint16), exactly as
    the GPU receives them.  Same outputs as :func:`sparse_mla_bwd_f64`."""
    return _bwd_f64(bf16_bits_to_f64(q_bits), bf16_bits_to_f64(kv_bits),
                    bf16_bits_to_f64(dout_bits), indices, topk_length, attn_sink, sm_scale,
                    threads, _lib_=_lib_)


# fixed references for BwdVariant (the pin tests rebind the public names to a variant)
_bwd_f64 = sparse_mla_bwd_f64
_bwd_bits = sparse_mla_bwd


class BwdVariant:
    """The backward bound to another build of its source (a shared library at ``path``); the
    pin tests use it to check that planted mistakes are caught."""

    def __init__(self, path):
        self._lib = _bind_bwd(ctypes.CDLL(path))

    def sparse_mla_bwd_f64(self, *a, **kw):
        return _bwd_f64(*a, _lib_=self._lib, **kw)

    def sparse_mla_bwd(self, *a, **kw):
        return _bwd_bits(*a, _lib_=self._lib, **kw)

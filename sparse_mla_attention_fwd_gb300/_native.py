"""ctypes view of the C ABI declared in include/sparse_mla.h.

Only argument marshalling happens here; every step of the forward runs in the CUDA library.
Loading fails loudly when the library has not been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .native_build import LIB_PATH

SMLA_OK = 0
STATUS_NAMES = {0: "SMLA_OK", 1: "SMLA_ERR_NULL_PTR", 2: "SMLA_ERR_BAD_SHAPE",
                3: "SMLA_ERR_MISALIGNED", 4: "SMLA_ERR_LAUNCH", 5: "SMLA_ERR_DEVICE_TIMEOUT",
                6: "SMLA_ERR_TENSOR_MAP", 7: "SMLA_ERR_WORKSPACE"}
EXPORTED = ("sparse_mla_fwd", "sparse_mla_fwd_paged", "sparse_mla_splitkv_workspace_size",
            "sparse_mla_fwd_splitkv", "sparse_mla_fwd_paged_splitkv", "sparse_mla_fwd_paged_splitkv_static",
            "sparse_mla_fwd_host", "sparse_mla_selftest_wait_timeout", "sparse_mla_device_status",
            "sparse_mla_status_string", "sparse_mla_abi_version", "sparse_mla_bwd")

_lock = threading.Lock()
_lib = None


class SmlaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)} ({status_string(code)})")


def load_library(path: str | None = None):
    """Load (once) and return the ctypes handle of the CUDA library."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library {path} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (no CPU fallback exists)")
        lib = ctypes.CDLL(path)
        P, I32, I64, F32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        lib.sparse_mla_fwd.restype = I32
        lib.sparse_mla_fwd.argtypes = [P, P, P, P, P, F32, I32, P, P, P, I64, I64, I32, I32, I32, P]
        lib.sparse_mla_fwd_paged.restype = I32
        lib.sparse_mla_fwd_paged.argtypes = [P, P, I64, P, I32, I32, P, I64, I32, P, P, P, F32, I32,
                                             P, P, P, I64, I32, I32, I32, P]
        SZ = ctypes.c_size_t
        lib.sparse_mla_splitkv_workspace_size.restype = SZ
        lib.sparse_mla_splitkv_workspace_size.argtypes = [I64, I32, I32]
        lib.sparse_mla_fwd_splitkv.restype = I32
        lib.sparse_mla_fwd_splitkv.argtypes = [P, P, P, P, P, F32, I32, P, P, P, I64, I64, I32, I32, I32,
                                               I32, P, SZ, P]
        lib.sparse_mla_fwd_paged_splitkv.restype = I32
        lib.sparse_mla_fwd_paged_splitkv.argtypes = [P, P, I64, P, I32, I32, P, I64, I32, P, P, P, F32, I32,
                                                     P, P, P, I64, I32, I32, I32, I32, P, SZ, P]
        lib.sparse_mla_fwd_paged_splitkv_static.restype = I32
        lib.sparse_mla_fwd_paged_splitkv_static.argtypes = [P, P, I64, P, I32, I32, P, I64, I32, P, P, P, F32,
                                                            I32, P, P, P, I64, I32, I32, I32, I32, P]
        lib.sparse_mla_fwd_host.restype = I32
        lib.sparse_mla_fwd_host.argtypes = [P, P, P, P, P, F32, I32, P, P, P, I64, I64, I32, I32, I32,
                                            P, P, P, P, P, P, P, P, I32, P, P, P]
        lib.sparse_mla_selftest_wait_timeout.restype = I32
        lib.sparse_mla_selftest_wait_timeout.argtypes = [ctypes.c_uint64, P]
        lib.sparse_mla_device_status.restype = I32
        lib.sparse_mla_device_status.argtypes = [I32]
        lib.sparse_mla_status_string.restype = ctypes.c_char_p
        lib.sparse_mla_status_string.argtypes = [I32]
        lib.sparse_mla_abi_version.restype = I32
        lib.sparse_mla_abi_version.argtypes = []
        lib.sparse_mla_bwd.restype = I32
        lib.sparse_mla_bwd.argtypes = [P, P, P, P, P, P, P, P, F32, I32, P, P, P, I64, I64, I32, I32, I32, P]
        _lib = lib
        return lib


def status_string(code: int) -> str:
    try:
        return load_library().sparse_mla_status_string(int(code)).decode()
    except RuntimeError:
        return STATUS_NAMES.get(code, "unknown")

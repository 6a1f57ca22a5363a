"""In-tree build of the CUDA library (sm_103a only).

``build()`` compiles ``csrc/sparse_mla_fwd.cu`` with nvcc into ``libsparse_mla_gb300.so`` next
to this file.  It is what ``__graft_entry__.build()`` runs on every machine (nvcc cross-compiles
without a GPU); the product path never compiles anything implicitly.
"""
from __future__ import annotations

import glob
import os
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
LIB_NAME = "libsparse_mla_gb300.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)
SOURCES = [os.path.join(PKG_DIR, "csrc", "sparse_mla_fwd.cu")]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _deps():
    return (SOURCES + glob.glob(os.path.join(PKG_DIR, "csrc", "*.cuh"))
            + glob.glob(os.path.join(ROOT, "include", "*.h")) + [os.path.abspath(__file__)])


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(d) > t for d in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not is_stale():
        return LIB_PATH
    nvcc = os.environ.get("NVCC", "nvcc")
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-o", tmp, *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))

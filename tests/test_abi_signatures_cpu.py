"""The ctypes binding and the C header agree: for every entry point that include/sparse_mla.h
declares, the binding sets a return type and one argument type per declared parameter, of the
matching kind (pointer, 32- or 64-bit integer, float, size).  A mismatch here would corrupt
arguments silently at run time, so it is checked without a GPU, from the header text."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sparse_mla.h")


def _declarations():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    decls = {}
    for m in re.finditer(r"([A-Za-z_][\w\s\*]*?)\b(sparse_mla_\w+)\s*\(([^;{]*?)\)\s*;", text):
        ret, name, params = m.group(1).strip(), m.group(2), m.group(3).strip()
        args = [] if params in ("", "void") else [p.strip() for p in params.split(",")]
        decls[name] = (ret, args)
    return decls


def _kind_of_c(decl):
    """Kind of a C parameter or return type: 'ptr', 'i32', 'i64', 'u64', 'f32', 'str' (size_t is
    64-bit unsigned on the LP64 hosts this runs on, so it counts as 'u64')."""
    d = " ".join(decl.replace("*", " * ").split())
    if "char *" in d and "const" in d:
        return "str"
    if "*" in d or "smla_stream_t" in d:
        return "ptr"
    t = d.split()
    base = [w for w in t[:-1] if w not in ("const",)] if len(t) > 1 else t
    base = " ".join(base) if base else d
    return {"int": "i32", "smla_status": "i32", "int64_t": "i64", "uint64_t": "u64", "float": "f32",
            "size_t": "u64"}.get(base, "?" + base)


def _kind_of_ctypes(t):
    if t in (ctypes.c_void_p,):
        return "ptr"
    if t is ctypes.c_char_p:
        return "str"
    if t is ctypes.c_float:
        return "f32"
    if issubclass(t, ctypes._SimpleCData):
        size, signed = ctypes.sizeof(t), t not in (ctypes.c_uint64, ctypes.c_uint32, ctypes.c_size_t)
        if size == 4:
            return "i32"
        if size == 8:
            return "i64" if signed else "u64"
    return "?" + t.__name__


@pytest.fixture(scope="module")
def lib():
    from sparse_mla_attention_fwd_gb300 import _native
    try:
        return _native.load_library()
    except RuntimeError as e:
        pytest.skip(str(e))


def test_header_parses_into_every_exported_entry_point():
    from sparse_mla_attention_fwd_gb300 import _native
    decls = _declarations()
    assert set(_native.EXPORTED) <= set(decls), sorted(set(_native.EXPORTED) - set(decls))


def test_binding_types_match_the_header(lib):
    from sparse_mla_attention_fwd_gb300 import _native
    decls = _declarations()
    for name in _native.EXPORTED:
        ret, args = decls[name]
        fn = getattr(lib, name)
        assert fn.argtypes is not None, f"{name}: no argtypes set"
        got = [_kind_of_ctypes(t) for t in fn.argtypes]
        want = [_kind_of_c(a.rsplit(" ", 1)[0] if not a.endswith("*") else a) for a in args]
        assert got == want, f"{name}: binding {got} vs header {want}"
        want_ret = _kind_of_c(ret)
        got_ret = _kind_of_ctypes(fn.restype) if fn.restype is not None else "?none"
        assert got_ret == want_ret, f"{name}: return {got_ret} vs {want_ret}"

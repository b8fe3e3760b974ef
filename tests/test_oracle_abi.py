"""The oracle's ctypes argument lists (oracle/__init__.py) match the C
definitions in oracle/oracle.c: the same count and, per position, a pointer,
a 32-bit int, a 64-bit int, a double, a float or a byte.  A mismatch would
not always fail a pin (a 64-bit value passed where 32 bits are read can still
work on one machine), so the signatures are checked directly."""
import ctypes
import os
import re

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _definitions():
    text = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    out = {}
    for m in re.finditer(r"^(int|void|double|uint8_t)\s+(oracle_\w+)\s*\(([^)]*)\)\s*\{",
                         text, flags=re.M):
        params = " ".join(m.group(3).split())
        out[m.group(2)] = (m.group(1),
                           [] if params in ("", "void") else [p.strip() for p in params.split(",")])
    return out


def _kind_c(param):
    if "*" in param:
        return "ptr"
    t = re.sub(r"\b\w+$", "", param).replace("const", "").strip()
    return {"int": "i32", "int64_t": "i64", "long": "i64", "double": "f64", "float": "f32",
            "uint8_t": "u8"}[t]


def _kind_py(a):
    if a is ctypes.c_void_p:
        return "ptr"
    return {ctypes.c_int: "i32", ctypes.c_int64: "i64", ctypes.c_double: "f64",
            ctypes.c_float: "f32", ctypes.c_uint8: "u8"}[a]


def test_oracle_signatures_match_the_c_definitions():
    lib = oracle._load()
    defs = _definitions()
    configured = [n for n in defs if getattr(lib, n).argtypes is not None]
    assert len(configured) >= 10
    returns = {"int": ctypes.c_int, "void": None, "double": ctypes.c_double,
               "uint8_t": ctypes.c_uint8}
    for name in configured:
        ret, params = defs[name]
        fn = getattr(lib, name)
        assert fn.restype is returns[ret], (name, ret, fn.restype)
        c_kinds = [_kind_c(p) for p in params]
        py_kinds = [_kind_py(a) for a in fn.argtypes]
        assert c_kinds == py_kinds, (name, c_kinds, py_kinds)

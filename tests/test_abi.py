"""The C ABI loads and exports every symbol include/pkx.h declares, and its
host-side argument checks reject bad calls before anything reaches a GPU.
(No compute call here: these run on a machine without a GPU.)"""
import ctypes
import os
import re

import pytest
import torch

from paged_kv_extend_gb300 import build as pkx_build
from paged_kv_extend_gb300 import pkx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkx.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkx_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    pkx_build.build()
    return pkx.load_library()


def test_header_declares_the_boundary():
    names = _declared()
    for must in ["pkx_extend_attention_fwd", "pkx_extend_attention_fwd_unified",
                 "pkx_decode_attention_fwd", "pkx_merge_state",
                 "pkx_build_unified_kv_indices", "pkx_extend_workspace_size",
                 "pkx_set_kv_buffer", "pkx_create_kv_indices", "pkx_set_kv_buffer_fp8",
                 "pkx_extend_attention_fwd_ragged_paged", "pkx_expand_paged_kv_indices",
                 "pkx_decode_workspace_size", "pkx_workspace_status",
                 "pkx_last_error_string", "pkx_version"]:
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    # and the binding knows the signature of each
    assert set(_declared()) == set(pkx._SIGS)


def test_version(lib):
    assert "sm_103a" in pkx.version()


def _extend(lib, **over):
    a = dict(q=None, k=None, v=None, o=None, kb=None, vb=None, qo=None, kvp=None, kvi=None,
             batch=1, n=4, hq=8, hkv=2, lq=128, lv=128, st=(1024, 128, 1024, 128, 1024, 128, 1024, 128),
             slots=16, scale=0.0, cap=0.0, win=-1, mask=None, mask_indptr=None, sinks=None,
             kvd=0, ksc=1.0, vsc=1.0, lse=None, ws=None, wsb=0, stream=None)
    a.update(over)
    return lib.pkx_extend_attention_fwd(
        a["q"], a["k"], a["v"], a["o"], a["kb"], a["vb"], a["qo"], a["kvp"], a["kvi"],
        a["batch"], a["n"], a["hq"], a["hkv"], a["lq"], a["lv"], *a["st"], a["slots"],
        a["scale"], a["cap"], a["win"], a["mask"], a["mask_indptr"], a["sinks"], a["kvd"],
        a["ksc"], a["vsc"], a["lse"], a["ws"], a["wsb"], a["stream"])


def _decode(lib, **over):
    a = dict(q=None, o=None, kb=None, vb=None, kvp=None, kvi=None, batch=1, hq=8, hkv=2, lq=128,
             lv=128, st=(1024, 128, 1024, 128), slots=16, scale=0.0, cap=0.0, win=-1, kvd=0,
             ksc=1.0, vsc=1.0, lse=None, ws=None, wsb=0, stream=None)
    a.update(over)
    return lib.pkx_decode_attention_fwd(
        a["q"], a["o"], a["kb"], a["vb"], a["kvp"], a["kvi"], a["batch"], a["hq"], a["hkv"],
        a["lq"], a["lv"], *a["st"], a["slots"], a["scale"], a["cap"], a["win"], a["kvd"],
        a["ksc"], a["vsc"], a["lse"], a["ws"], a["wsb"], a["stream"])


def test_host_validation_rejects_bad_arguments(lib):
    assert _extend(lib, hq=6, hkv=4) == pkx.PKX_EINVAL
    assert b"multiple" in lib.pkx_last_error_string()
    assert _extend(lib, lq=96, lv=96) == pkx.PKX_EUNSUPPORTED
    # the split head dims pass the head check (the null q is what is refused)
    assert _extend(lib, lq=192, lv=128) == pkx.PKX_EINVAL
    assert b"q_extend" in lib.pkx_last_error_string()
    assert _extend(lib, lq=288, lv=256, hq=16, hkv=1) == pkx.PKX_EINVAL
    assert _extend(lib, lq=192, lv=256) == pkx.PKX_EUNSUPPORTED
    assert b"lq=192" in lib.pkx_last_error_string()
    # an fp8 pool with the split head dims is built for extend (past the
    # format check, the null tensors stop the call), not for decode
    assert _extend(lib, lq=192, lv=128, kvd=1) == pkx.PKX_EINVAL
    assert b"q_extend" in lib.pkx_last_error_string()
    assert _decode(lib, lq=192, lv=128, kvd=1) == pkx.PKX_EUNSUPPORTED
    assert _decode(lib, lq=288, lv=256, hq=16, hkv=1, kvd=2) == pkx.PKX_EUNSUPPORTED
    assert _decode(lib, kvd=1) == pkx.PKX_EINVAL  # D = 128: built, null tensors
    assert _extend(lib, hq=256, hkv=1) == pkx.PKX_EUNSUPPORTED
    assert _extend(lib, batch=-1) == pkx.PKX_EINVAL
    assert _extend(lib, scale=float("nan")) == pkx.PKX_EINVAL
    # a custom mask needs its offsets; sinks must be aligned
    assert _extend(lib, mask=0x1000) == pkx.PKX_EINVAL
    assert b"mask_indptr" in lib.pkx_last_error_string()
    assert _extend(lib, sinks=0x1002) == pkx.PKX_EINVAL
    # null tensors
    assert _extend(lib) == pkx.PKX_EINVAL
    assert b"null" in lib.pkx_last_error_string()
    # misaligned pointer (never dereferenced: validation fails first)
    assert _extend(lib, q=0x1008) == pkx.PKX_EINVAL
    # stride not a multiple of 8 elements
    assert _extend(lib, q=0x1000, o=0x1000, k=0x1000, v=0x1000, kb=0x1000, vb=0x1000,
                   st=(1024, 127, 1024, 128, 1024, 128, 1024, 128)) == pkx.PKX_EINVAL
    # pool format: an unknown format, bad scales, fp8 where it is not built
    assert _extend(lib, kvd=3) == pkx.PKX_EINVAL
    assert _extend(lib, kvd=1, ksc=0.0) == pkx.PKX_EINVAL
    assert _extend(lib, kvd=2, vsc=float("inf")) == pkx.PKX_EINVAL
    assert _extend(lib, kvd=1, lq=96, lv=96) == pkx.PKX_EUNSUPPORTED
    # the MLA head over an fp8 pool is built: past the format check, the null
    # tensors stop the call
    assert _extend(lib, kvd=1, lq=576, lv=512, hq=16, hkv=1) == pkx.PKX_EINVAL
    assert b"fp8" not in lib.pkx_last_error_string()
    # a custom mask over an fp8 pool is built: the call gets past the format
    # check and stops at the null tensors
    assert _extend(lib, kvd=1, mask=0x1000, mask_indptr=0x1000) == pkx.PKX_EINVAL
    assert b"fp8" not in lib.pkx_last_error_string()
    # empty problem: nothing to do, succeeds without touching a device
    assert _extend(lib, batch=0) == pkx.PKX_OK
    assert _extend(lib, n=0) == pkx.PKX_OK


def test_merge_and_index_validation(lib):
    assert lib.pkx_merge_state(None, None, None, None, None, None, 4, 2, 12, None) == pkx.PKX_EINVAL
    assert lib.pkx_merge_state(None, None, None, None, None, None, 4, 2, 16, None) == pkx.PKX_EINVAL
    assert lib.pkx_merge_state(None, None, None, None, None, None, 0, 2, 16, None) == pkx.PKX_OK
    assert lib.pkx_build_unified_kv_indices(None, None, None, None, None, 3, None, None, None,
                                            None) == pkx.PKX_EINVAL
    assert lib.pkx_workspace_status(None, None) == pkx.PKX_EINVAL


def test_fp8_write_validation(lib):
    A = 0x10000
    w = lambda **o: lib.pkx_set_kv_buffer_fp8(
        A, 256, 128, A, 256, 128, A, o.get("n", 4), 2, 128, 128, o.get("ks", 1.0),
        o.get("vs", 1.0), o.get("fmt", 1), A, 256, 128, A, 256, 128, 64, None)
    assert w(fmt=0) == pkx.PKX_EINVAL        # bf16 is not an fp8 format
    assert w(fmt=3) == pkx.PKX_EINVAL
    assert w(ks=-1.0) == pkx.PKX_EINVAL
    assert w(vs=float("nan")) == pkx.PKX_EINVAL
    assert w(n=0) == pkx.PKX_OK
    assert w(n=0, fmt=2) == pkx.PKX_OK


def test_paged_expansion_validation(lib):
    A = 0x10000
    e = lambda **o: lib.pkx_expand_paged_kv_indices(
        o.get("ptr", A), A, o.get("last", A), o.get("ps", 16), o.get("bs", 2), o.get("out", A),
        A, o.get("cap", 64), None)
    assert e(ps=0) == pkx.PKX_EINVAL
    assert e(bs=12001) == pkx.PKX_EUNSUPPORTED
    assert e(out=None) == pkx.PKX_EINVAL
    assert e(last=A + 2) == pkx.PKX_EINVAL
    assert e(ptr=None) == pkx.PKX_EINVAL
    assert e(cap=-1) == pkx.PKX_EINVAL


def test_kv_write_and_gather_validation(lib):
    """pkx_set_kv_buffer / pkx_create_kv_indices reject bad arguments on the
    host (and an empty call is a no-op that needs no device)."""
    A = 0x10000  # an aligned stand-in pointer; never dereferenced on these paths
    kv = lambda **o: lib.pkx_set_kv_buffer(
        o.get("k", A), o.get("kts", 256), 128, o.get("v", A), 256, 128, o.get("loc", A),
        o.get("n", 4), 2, o.get("lk", 128), o.get("lv", 128), o.get("kb", A), 256, 128, A,
        256, 128, 64, None)
    assert kv(n=0) == pkx.PKX_OK
    assert kv(lk=100) == pkx.PKX_EINVAL          # not a multiple of 8
    assert kv(lv=0) == pkx.PKX_EINVAL
    assert kv(loc=None) == pkx.PKX_EINVAL
    assert kv(loc=A + 4) == pkx.PKX_EINVAL       # int64 misaligned
    assert kv(k=A + 2) == pkx.PKX_EINVAL         # bf16 rows must be 16-byte aligned
    assert kv(kts=260) == pkx.PKX_EINVAL         # stride not a multiple of 8
    assert kv(kb=None) == pkx.PKX_EINVAL
    assert kv(v=None, lv=0, n=0) == pkx.PKX_OK   # K-only pool
    g = lambda **o: lib.pkx_create_kv_indices(
        o.get("rt", A), 4, 8, o.get("rpi", A), o.get("lens", A), o.get("start", None),
        o.get("bs", 2), o.get("ptr", A), o.get("idx", A), o.get("cap", 16), None)
    assert g(bs=-1) == pkx.PKX_EUNSUPPORTED
    assert g(bs=12001) == pkx.PKX_EUNSUPPORTED
    assert g(ptr=None) == pkx.PKX_EINVAL
    assert g(ptr=A + 2) == pkx.PKX_EINVAL
    assert g(rpi=None) == pkx.PKX_EINVAL
    assert g(lens=A + 4) == pkx.PKX_EINVAL
    assert g(start=A + 4) == pkx.PKX_EINVAL
    assert g(idx=None) == pkx.PKX_EINVAL
    assert g(rt=None) == pkx.PKX_EINVAL
    assert g(cap=-1) == pkx.PKX_EINVAL


def test_workspace_size_grows_with_problem(lib):
    a = pkx.extend_workspace_size(16, 9000, 32, 8, 128, 128)
    b = pkx.extend_workspace_size(64, 1024, 32, 8, 128, 128)
    assert a > 0 and b > 0
    assert pkx.extend_workspace_size(16, 90000, 32, 8, 128, 128) > a
    assert pkx.extend_workspace_size(16, 9000, 30, 8, 128, 128) == 0  # hq % hkv != 0
    assert pkx.decode_workspace_size(64, 32, 8, 128, 128) > 0


def test_workspace_size_relations(lib):
    """Host-side sizing the calls rely on: the one-stream decode layout never
    exceeds the two-stream one (the call falls back to it), the ragged +
    paged split holds at least one extend pass's scratch, and sizes grow
    with the problem."""
    for hq, hkv, d in [(32, 8, 128), (16, 16, 64), (28, 4, 128), (64, 8, 64), (16, 1, 576)]:
        lv = 512 if d == 576 else d
        prev = 0
        for b in (1, 7, 64, 1000, 4096):
            full = pkx.decode_workspace_size(b, hq, hkv, d, lv)
            small = pkx.decode_workspace_min_size(b, hq, hkv, d, lv)
            assert 0 < small <= full
            assert full >= prev
            prev = full
        for b, n in ((1, 1), (16, 8353), (256, 100000)):
            ext = pkx.extend_workspace_size(b, n, hq, hkv, d, lv)
            split = pkx.ragged_paged_workspace_size(b, n, hq, hkv, d, lv)
            assert 0 < ext < split
    assert pkx.decode_workspace_min_size(4, 30, 8, 128, 128) == 0  # hq % hkv != 0


def test_plain_c_consumer(lib, tmp_path):
    """pkx.h compiles as strict C99 and C++11, and a C program linked against
    libpkx.so gets the version, workspace sizes and host-side rejections
    without Python in between."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None or shutil.which("g++") is None:
        pytest.skip("no host C compiler")
    libdir = os.path.dirname(pkx.LIB_PATH)
    exe = str(tmp_path / "c_consumer")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_consumer.c"),
                    "-L", libdir, "-lpkx", "-Wl,-rpath," + libdir, "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.startswith("ok ") and "sm_103a" in r.stdout
    cxx = tmp_path / "header.cpp"
    cxx.write_text('#include "pkx.h"\nint main() { return pkx_version() == nullptr; }\n')
    subprocess.run(["g++", "-std=c++11", "-Wall", "-Werror", "-pedantic", "-fsyntax-only",
                    "-I", os.path.join(ROOT, "include"), str(cxx)], check=True)


def test_header_constants_match_the_binding():
    """Every status code and pool-format value pkx.h defines has the same
    value in the Python binding."""
    text = open(HEADER).read()
    defs = dict(re.findall(r"#define (PKX_\w+) (\d+)", text))
    assert {"PKX_OK", "PKX_EINVAL", "PKX_EWORKSPACE", "PKX_KV_BF16", "PKX_KV_FP8_E5M2"} <= set(defs)
    for name, value in defs.items():
        assert getattr(pkx, name) == int(value), name


def _prototypes():
    """name -> list of parameter C types, from pkx.h (comments removed)."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    protos = {}
    for m in re.finditer(r"\b(pkx_\w+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        params = " ".join(m.group(2).split())
        if params in ("", "void"):
            protos[m.group(1)] = []
            continue
        types = []
        for p in params.split(","):
            p = p.strip()
            # drop the parameter name: the last identifier, unless it is all there is
            ptype = re.sub(r"\b\w+$", "", p).strip() if re.search(r"[\s*]\w+$", p) else p
            types.append(ptype)
        protos[m.group(1)] = types
    return protos


def test_binding_signatures_match_the_header():
    """The ctypes argument list of every entry point matches its C prototype:
    the same count, and per position a pointer, a 32-bit int, a 64-bit int,
    a size_t or a float."""
    import ctypes

    def kind_c(t):
        if "*" in t:
            return "ptr"
        t = t.replace("const", "").strip()
        # uint64_t and size_t are both 64-bit unsigned here (ctypes has one type)
        return {"int": "i32", "int64_t": "i64", "size_t": "size", "uint64_t": "size",
                "float": "f32"}[t]

    def kind_py(a):
        if a in (ctypes.c_void_p, ctypes.c_char_p):
            return "ptr"
        if a is ctypes.c_size_t:
            return "size"
        return {ctypes.c_int: "i32", ctypes.c_int64: "i64", ctypes.c_float: "f32"}[a]

    protos = _prototypes()
    assert set(protos) == set(pkx._SIGS)
    for name, (_, args) in pkx._SIGS.items():
        c_kinds = [kind_c(t) for t in protos[name]]
        py_kinds = [kind_py(a) for a in args]
        assert c_kinds == py_kinds, (name, c_kinds, py_kinds)


def test_binding_refuses_host_tensors():
    """A host tensor among the arguments never reaches the library (it would
    arrive in a kernel as a host address): the binding raises first."""
    v = torch.zeros(4, 2, 16, dtype=torch.bfloat16)
    s = torch.zeros(4, 2, dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA"):
        pkx.merge_state(v, s, v, s)
    with pytest.raises(ValueError, match="CUDA"):
        pkx._ptr(s)
    assert pkx._ptr(None) is None


def test_binding_checks_shapes_before_the_call():
    """An output smaller than the problem, or index arrays of the wrong
    length, are refused in the binding (the C entry points take raw
    pointers and would write out of bounds).  Host tensors are enough here:
    the shape checks come before any pointer is taken."""
    bf = torch.bfloat16
    q = torch.zeros(5, 8, 128, dtype=bf)
    kb = torch.zeros(64, 2, 128, dtype=bf)
    kvp = torch.zeros(3, dtype=torch.int32)
    kvi = torch.zeros(0, dtype=torch.int32)
    with pytest.raises(ValueError, match="o has shape"):
        pkx.decode_attention_fwd(q, torch.zeros(5, 8, 64, dtype=bf), kb, kb, kvp, kvi)
    with pytest.raises(ValueError, match="lse"):
        pkx.decode_attention_fwd(q, torch.zeros_like(q), kb, kb, kvp, kvi,
                                 lse=torch.zeros(5, 4))
    with pytest.raises(ValueError, match="kv_indptr has 3 entries, expected 6"):
        pkx.decode_attention_fwd(q, torch.zeros_like(q), kb, kb, kvp, kvi)
    with pytest.raises(ValueError, match="disagree"):
        pkx.decode_attention_fwd(q, torch.zeros_like(q), kb, torch.zeros(32, 2, 128, dtype=bf),
                                 torch.zeros(6, dtype=torch.int32), kvi)
    with pytest.raises(ValueError, match="k_extend"):
        pkx.extend_attention_fwd(q, torch.zeros(4, 2, 128, dtype=bf), torch.zeros(5, 2, 128, dtype=bf),
                                 torch.zeros_like(q), kb, kb, torch.zeros(2, dtype=torch.int32),
                                 torch.zeros(2, dtype=torch.int32), kvi)
    v = torch.zeros(4, 2, 16, dtype=bf)
    with pytest.raises(ValueError, match="v_a's shape"):
        pkx.merge_state(v, torch.zeros(4, 2), torch.zeros(4, 2, 8, dtype=bf), torch.zeros(4, 2))

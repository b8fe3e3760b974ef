"""The C ABI loads and exports every symbol include/pkx.h declares, and its
host-side argument checks reject bad calls before anything reaches a GPU.
(No compute call here: these run on a machine without a GPU.)"""
import ctypes
import os
import re

import pytest

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
             lse=None, ws=None, wsb=0, stream=None)
    a.update(over)
    return lib.pkx_extend_attention_fwd(
        a["q"], a["k"], a["v"], a["o"], a["kb"], a["vb"], a["qo"], a["kvp"], a["kvi"],
        a["batch"], a["n"], a["hq"], a["hkv"], a["lq"], a["lv"], *a["st"], a["slots"],
        a["scale"], a["cap"], a["win"], a["mask"], a["mask_indptr"], a["sinks"], a["lse"],
        a["ws"], a["wsb"], a["stream"])


def test_host_validation_rejects_bad_arguments(lib):
    assert _extend(lib, hq=6, hkv=4) == pkx.PKX_EINVAL
    assert b"multiple" in lib.pkx_last_error_string()
    assert _extend(lib, lq=96, lv=96) == pkx.PKX_EUNSUPPORTED
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


def test_workspace_size_grows_with_problem(lib):
    a = pkx.extend_workspace_size(16, 9000, 32, 8, 128, 128)
    b = pkx.extend_workspace_size(64, 1024, 32, 8, 128, 128)
    assert a > 0 and b > 0
    assert pkx.extend_workspace_size(16, 90000, 32, 8, 128, 128) > a
    assert pkx.extend_workspace_size(16, 9000, 30, 8, 128, 128) == 0  # hq % hkv != 0
    assert pkx.decode_workspace_size(64, 32, 8, 128, 128) > 0

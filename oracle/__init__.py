"""Float64 CPU oracle for paged-KV extend attention and its companions.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product library (``paged_kv_extend_gb300``) never imports, loads or calls it,
and this package imports nothing from the product library.

The arithmetic lives in ``oracle.c`` (plain C, double precision, loops over
sequence -> head -> query -> key).  This module only compiles it with gcc and
marshals torch CPU tensors into it.  Each wrapper names the page section whose
definition it restates; the C file states the definition itself.

Pins: every function here is checked against something other than itself in
``tests/test_oracle_pins.py`` (library routines, closed forms, invariants the
pages fix, and hand-derived golden values under ``tests/golden/``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_p = ctypes.c_void_p
_l = ctypes.c_long
_i = ctypes.c_int
_d = ctypes.c_double


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, -O2, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _configure(lib):
    lib.oracle_num_threads.restype = _i
    lib.oracle_extend_attention.restype = _i
    lib.oracle_extend_attention.argtypes = [
        _p, _p, _l, _l, _p, _l, _l, _p, _l, _l, _p, _l, _l, _i, _d, _d,
        _p, _p, _p, _i, _i, _i, _i, _i, _d, _d, _l, _p, _p, _p, _p, _l, _p, _p]
    lib.oracle_extend_attention_unified.restype = _i
    lib.oracle_extend_attention_unified.argtypes = [
        _p, _p, _l, _l, _p, _l, _l, _i, _d, _d, _p, _p, _p, _p,
        _i, _i, _i, _i, _i, _d, _d, _l, _p, _p, _p, _p, _l, _p, _p]
    lib.oracle_decode_attention.restype = _i
    lib.oracle_decode_attention.argtypes = [
        _p, _p, _l, _l, _p, _l, _l, _i, _d, _d, _p, _p,
        _i, _i, _i, _i, _i, _d, _d, _l, _p, _p]
    lib.oracle_merge_state.restype = None
    lib.oracle_merge_state.argtypes = [_p, _p, _p, _p, _l, _i, _i, _p, _p]
    lib.oracle_build_unified_kv_indices.restype = None
    lib.oracle_build_unified_kv_indices.argtypes = [
        _p, _p, _p, _p, _p, _i, _p, _p, _p]
    lib.oracle_create_kv_indices.restype = None
    lib.oracle_create_kv_indices.argtypes = [_p, _l, _p, _p, _p, _i, _p, _p]
    lib.oracle_fp8_value.restype = _d
    lib.oracle_fp8_value.argtypes = [ctypes.c_uint8, _i]
    lib.oracle_fp8_code.restype = ctypes.c_uint8
    lib.oracle_fp8_code.argtypes = [ctypes.c_float, _i]
    lib.oracle_set_kv_buffer_fp8.restype = None
    lib.oracle_set_kv_buffer_fp8.argtypes = [
        _p, _l, _l, _p, _l, _l, _p, _l, _i, _i, _i, ctypes.c_float, ctypes.c_float, _i,
        _p, _l, _l, _p, _l, _l]
    lib.oracle_expand_paged_kv_indices.restype = None
    lib.oracle_expand_paged_kv_indices.argtypes = [_p, _p, _p, _i, _i, _p, _p]
    lib.oracle_set_kv_buffer.restype = None
    lib.oracle_set_kv_buffer.argtypes = [
        _p, _l, _l, _p, _l, _l, _p, _l, _i, _i, _i, _p, _l, _l, _p, _l, _l]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
    return _lib


class use_library:
    """Context manager for tests: run the wrappers against another build of
    the oracle (e.g. one with a deliberately planted mistake)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        _load()
        self._saved = _lib
        _lib = None
        _lib = _configure(ctypes.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def num_threads() -> int:
    """OpenMP threads the oracle runs on."""
    return int(_load().oracle_num_threads())


# ---------------------------------------------------------------- marshalling
def _bf16_bits(t: torch.Tensor) -> torch.Tensor:
    """A CPU bf16 tensor reinterpreted as its int16 bit patterns (no copy of
    values, strides preserved)."""
    assert t.dtype == torch.bfloat16, t.dtype
    return t.detach().cpu().view(torch.int16)


def _ptr(t) -> int:
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _i32(t: torch.Tensor) -> torch.Tensor:
    return t.detach().cpu().to(torch.int32).contiguous()


def _i64(t: torch.Tensor) -> torch.Tensor:
    return t.detach().cpu().to(torch.int64).contiguous()


def _row_strides(t: torch.Tensor):
    """(token/slot stride, head stride) in elements of a [n, h, d] view whose
    last dim is contiguous."""
    assert t.dim() == 3 and t.stride(2) == 1, (t.shape, t.stride())
    return t.stride(0), t.stride(1)


def _rows_arg(rows):
    if rows is None:
        return None, 0
    r = _i64(torch.as_tensor(rows))
    return r, r.numel()


def _mask_args(custom_mask, mask_indptr, sinks, hq):
    """(custom_mask uint8, mask_indptr int32, sinks float64) tensors or None;
    a custom mask needs its offsets, sinks are one logit per query head."""
    cm = mi = sk = None
    if custom_mask is not None:
        if mask_indptr is None:
            raise ValueError("custom_mask needs mask_indptr")
        cm = torch.as_tensor(custom_mask).to(torch.uint8).contiguous().cpu()
        mi = _i32(mask_indptr)
    if sinks is not None:
        sk = torch.as_tensor(sinks).to(torch.float64).contiguous().cpu()
        if sk.numel() != hq:
            raise ValueError("sinks must hold one value per query head")
    return cm, mi, sk


# pool element formats (oracle.c KV_BF16 / KV_E4M3 / KV_E5M2)
KV_BF16, KV_E4M3, KV_E5M2 = 0, 1, 2
_FP8 = {KV_E4M3: torch.float8_e4m3fn, KV_E5M2: torch.float8_e5m2}


def _pool(t: torch.Tensor):
    """(element view for the C side, format) of a bf16 or fp8 pool tensor."""
    if t.dtype == torch.bfloat16:
        return _bf16_bits(t), KV_BF16
    for fmt, dt in _FP8.items():
        if t.dtype == dt:
            return t.detach().cpu().view(torch.uint8), fmt
    raise ValueError(f"pool dtype {t.dtype} is neither bf16 nor fp8")


def _pools(k_buffer, v_buffer):
    kb, fk = _pool(k_buffer)
    vb, fv = _pool(v_buffer)
    if fk != fv:
        raise ValueError("k_buffer and v_buffer must share one format")
    return kb, vb, fk


def _opt(t):
    return _ptr(t) if t is not None and t.numel() else None


# ------------------------------------------------------------------ functions
def extend_attention(q_extend, k_extend, v_extend, k_buffer, v_buffer,
                     qo_indptr, kv_indptr, kv_indices, sm_scale, logit_cap=0.0,
                     sliding_window=-1, rows=None, custom_mask=None, mask_indptr=None,
                     sinks=None, k_scale=1.0, v_scale=1.0):
    """Two-stage extend attention (sglang extend_attention.py,
    extend_attention_fwd): prefix K/V through kv_indptr/kv_indices into the
    pool, extend K/V contiguous at qo_indptr.

    custom_mask (bytes, row i of sequence b at mask_indptr[b] + i * T_b over
    its T_b keys) replaces the causal mask; sinks [Hq] add exp(sink - m) to
    each row's softmax denominator (sglang extend_attention.py,
    _fwd_kernel_unified).

    q_extend [N, Hq, Lq] bf16; k_extend [N, Hkv, Lq]; v_extend [N, Hkv, Lv];
    k_buffer [S, Hkv, Lq]; v_buffer [S, Hkv, Lv] (views with a contiguous last
    dim; v may alias k).  sm_scale <= 0 means 1/sqrt(Lq).  The pool may be
    fp8 (torch.float8_e4m3fn / float8_e5m2): its keys then read code *
    k_scale and its values code * v_scale (sglang flashinfer_backend.py,
    forward with k_scale / v_scale).
    Returns (o [N, Hq, Lv] float64, lse [N, Hq] float64), or for ``rows`` (a
    list of token*Hq + head) o [R, Lv] and lse [R].
    """
    lib = _load()
    n, hq, lq = q_extend.shape
    hkv = k_buffer.shape[1]
    lv = v_buffer.shape[2]
    if sm_scale is None or sm_scale <= 0:
        sm_scale = 1.0 / (lq ** 0.5)
    q = _bf16_bits(q_extend).contiguous()
    ke, ve = _bf16_bits(k_extend), _bf16_bits(v_extend)
    kb, vb, fmt = _pools(k_buffer, v_buffer)
    qo, kvp, kvi = _i32(qo_indptr), _i32(kv_indptr), _i32(kv_indices)
    batch = qo.numel() - 1
    cm, mi, sk = _mask_args(custom_mask, mask_indptr, sinks, hq)
    rws, nr = _rows_arg(rows)
    count = nr if rws is not None else n * hq
    o = torch.empty(count, lv, dtype=torch.float64)
    lse = torch.empty(count, dtype=torch.float64)
    rc = lib.oracle_extend_attention(
        _ptr(q), _ptr(ke), *_row_strides(ke), _ptr(ve), *_row_strides(ve),
        _ptr(kb), *_row_strides(kb), _ptr(vb), *_row_strides(vb),
        fmt, float(k_scale), float(v_scale),
        _ptr(qo), _ptr(kvp), _ptr(kvi) if kvi.numel() else None,
        batch, hq, hkv, lq, lv, float(sm_scale), float(logit_cap),
        int(sliding_window), _opt(cm), _opt(mi), _opt(sk),
        _ptr(rws) if rws is not None else None, nr, _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_extend_attention: bad arguments")
    if rws is None:
        return o.view(n, hq, lv), lse.view(n, hq)
    return o, lse


def extend_attention_unified(q, k_buffer, v_buffer, qo_indptr, kv_indptr,
                             kv_indices, prefix_lens, sm_scale, logit_cap=0.0,
                             sliding_window=-1, rows=None, custom_mask=None,
                             mask_indptr=None, sinks=None, k_scale=1.0, v_scale=1.0):
    """Unified extend attention (sglang extend_attention.py,
    extend_attention_fwd_unified): all keys through the unified int64
    kv_indices; the first prefix_lens[b] keys of sequence b are its prefix.
    Shapes and returns as :func:`extend_attention`."""
    lib = _load()
    n, hq, lq = q.shape
    hkv = k_buffer.shape[1]
    lv = v_buffer.shape[2]
    if sm_scale is None or sm_scale <= 0:
        sm_scale = 1.0 / (lq ** 0.5)
    qb = _bf16_bits(q).contiguous()
    kb, vb, fmt = _pools(k_buffer, v_buffer)
    qo, kvp, kvi, pl = _i32(qo_indptr), _i32(kv_indptr), _i64(kv_indices), _i32(prefix_lens)
    batch = qo.numel() - 1
    cm, mi, sk = _mask_args(custom_mask, mask_indptr, sinks, hq)
    rws, nr = _rows_arg(rows)
    count = nr if rws is not None else n * hq
    o = torch.empty(count, lv, dtype=torch.float64)
    lse = torch.empty(count, dtype=torch.float64)
    rc = lib.oracle_extend_attention_unified(
        _ptr(qb), _ptr(kb), *_row_strides(kb), _ptr(vb), *_row_strides(vb),
        fmt, float(k_scale), float(v_scale),
        _ptr(qo), _ptr(kvp), _ptr(kvi) if kvi.numel() else None, _ptr(pl),
        batch, hq, hkv, lq, lv, float(sm_scale), float(logit_cap),
        int(sliding_window), _opt(cm), _opt(mi), _opt(sk),
        _ptr(rws) if rws is not None else None, nr, _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_extend_attention_unified: bad arguments")
    if rws is None:
        return o.view(n, hq, lv), lse.view(n, hq)
    return o, lse


def decode_attention(q, k_buffer, v_buffer, kv_indptr, kv_indices, sm_scale,
                     logit_cap=0.0, sliding_window=-1, k_scale=1.0, v_scale=1.0):
    """Decode attention (sglang flashinfer_backend.py, forward_decode): one
    query per sequence over all of its pooled keys.
    q [B, Hq, Lq] bf16 -> (o [B, Hq, Lv] float64, lse [B, Hq] float64)."""
    lib = _load()
    b, hq, lq = q.shape
    hkv = k_buffer.shape[1]
    lv = v_buffer.shape[2]
    if sm_scale is None or sm_scale <= 0:
        sm_scale = 1.0 / (lq ** 0.5)
    qb = _bf16_bits(q).contiguous()
    kb, vb, fmt = _pools(k_buffer, v_buffer)
    kvp, kvi = _i32(kv_indptr), _i32(kv_indices)
    o = torch.empty(b, hq, lv, dtype=torch.float64)
    lse = torch.empty(b, hq, dtype=torch.float64)
    rc = lib.oracle_decode_attention(
        _ptr(qb), _ptr(kb), *_row_strides(kb), _ptr(vb), *_row_strides(vb),
        fmt, float(k_scale), float(v_scale), _ptr(kvp),
        _ptr(kvi) if kvi.numel() else None, b, hq, hkv, lq, lv,
        float(sm_scale), float(logit_cap), int(sliding_window), _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_decode_attention: bad arguments")
    return o, lse


def merge_state(v_a, s_a, v_b, s_b):
    """merge_state (sglang flashinfer_backend.py, forward_extend ragged +
    paged split).  v_* [N, H, Dv] bf16, s_* [N, H] fp32 ->
    (v [N, H, Dv] float64, s [N, H] float64)."""
    lib = _load()
    n, h, dv = v_a.shape
    va, vb = _bf16_bits(v_a).contiguous(), _bf16_bits(v_b).contiguous()
    sa = s_a.detach().cpu().to(torch.float32).contiguous()
    sb = s_b.detach().cpu().to(torch.float32).contiguous()
    v = torch.empty(n, h, dv, dtype=torch.float64)
    s = torch.empty(n, h, dtype=torch.float64)
    lib.oracle_merge_state(_ptr(va), _ptr(sa), _ptr(vb), _ptr(sb), n, h, dv,
                           _ptr(v), _ptr(s))
    return v, s


def build_unified_kv_indices(prefix_kv_indptr, prefix_kv_indices,
                             extend_start_loc, extend_seq_lens,
                             extend_kv_indices, bs, fill=-1):
    """Unified KV-index build (sglang extend_attention.py,
    build_unified_kv_indices).  Returns (unified_kv_indptr int32 [bs+1],
    unified_kv_indices int64 [len(prefix)+len(extend)], prefix_lens int32
    [bs]); entries past unified_kv_indptr[bs] keep the value ``fill``."""
    lib = _load()
    pip, pix = _i32(prefix_kv_indptr), _i32(prefix_kv_indices)
    esl, eln, eix = _i32(extend_start_loc), _i32(extend_seq_lens), _i32(extend_kv_indices)
    uptr = torch.empty(bs + 1, dtype=torch.int32)
    uidx = torch.full((pix.numel() + eix.numel(),), fill, dtype=torch.int64)
    plen = torch.empty(bs, dtype=torch.int32)
    lib.oracle_build_unified_kv_indices(
        _ptr(pip), _ptr(pix) if pix.numel() else None, _ptr(esl), _ptr(eln),
        _ptr(eix) if eix.numel() else None, int(bs), _ptr(uptr),
        _ptr(uidx) if uidx.numel() else None, _ptr(plen))
    return uptr, uidx, plen


def create_kv_indices(req_to_token, req_pool_indices, paged_kernel_lens,
                      kv_start_idx=None, fill=-1):
    """KV-index gather (sglang flashinfer_backend.py,
    create_flashinfer_kv_indices_triton and its callers' indptr).
    req_to_token int32 [R, C]; req_pool_indices, paged_kernel_lens,
    kv_start_idx int64 [bs].  Returns (kv_indptr int32 [bs+1], kv_indices
    int32 [sum(paged_kernel_lens)]); ``fill`` marks entries not written."""
    lib = _load()
    rt = req_to_token.detach().cpu().to(torch.int32).contiguous()
    rpi, pkl = _i64(req_pool_indices), _i64(paged_kernel_lens)
    kst = _i64(kv_start_idx) if kv_start_idx is not None else None
    bs = rpi.numel()
    total = int(pkl.to(torch.int32).sum()) if bs else 0
    kvp = torch.empty(bs + 1, dtype=torch.int32)
    kvi = torch.full((total,), fill, dtype=torch.int32)
    lib.oracle_create_kv_indices(
        _ptr(rt) if rt.numel() else None, rt.shape[1] if rt.dim() == 2 else 0,
        _ptr(rpi) if bs else None, _ptr(pkl) if bs else None,
        _ptr(kst) if kst is not None and bs else None, bs, _ptr(kvp),
        _ptr(kvi) if total else None)
    return kvp, kvi


def set_kv_buffer(k_buffer, v_buffer, cache_loc, k, v):
    """KV write into the pool (sglang flashinfer_backend.py, set_kv_buffer
    before the paged pass).  Returns new (k_buffer, v_buffer) bf16 tensors
    equal to the inputs with row cache_loc[t] of every KV head replaced by
    k[t] / v[t]; ``v`` may be None (K-only pool: v_buffer returned as is)."""
    lib = _load()
    kb = _bf16_bits(k_buffer).clone().contiguous()
    vb = _bf16_bits(v_buffer).clone().contiguous()
    kk = _bf16_bits(k).contiguous()
    vv = _bf16_bits(v).contiguous() if v is not None else None
    loc = _i64(cache_loc)
    n, hkv, lk = kk.shape
    lv = vv.shape[2] if vv is not None else 0
    lib.oracle_set_kv_buffer(
        _ptr(kk), *_row_strides(kk), _ptr(vv) if vv is not None else None,
        *(_row_strides(vv) if vv is not None else (0, 0)),
        _ptr(loc) if n else None, n, hkv, lk, lv,
        _ptr(kb), *_row_strides(kb), _ptr(vb), *_row_strides(vb))
    return kb.view(torch.bfloat16), vb.view(torch.bfloat16)


def fp8_value(code: int, fmt: int) -> float:
    """The value of one fp8 code (fmt KV_E4M3 or KV_E5M2)."""
    return float(_load().oracle_fp8_value(int(code) & 0xFF, int(fmt)))


def fp8_code(x: float, fmt: int) -> int:
    """The fp8 code of an fp32 value: nearest, ties to even, saturating."""
    return int(_load().oracle_fp8_code(float(x), int(fmt)))


def set_kv_buffer_fp8(k_buffer, v_buffer, cache_loc, k, v, k_scale, v_scale):
    """KV write into an fp8 pool (sglang flashinfer_backend.py,
    set_kv_buffer(layer, cache_loc, k, v, k_scale, v_scale) with an fp8 KV
    cache): every element of k[t] / v[t] divided by its scale in fp32 and
    stored as its nearest fp8 code at slot cache_loc[t].  Pools are
    torch.float8_e4m3fn or float8_e5m2; returns new (k_buffer, v_buffer)."""
    lib = _load()
    kb0, vb0, fmt = _pools(k_buffer, v_buffer)
    if fmt == KV_BF16:
        raise ValueError("set_kv_buffer_fp8 needs an fp8 pool")
    kb, vb = kb0.clone().contiguous(), vb0.clone().contiguous()
    kk = _bf16_bits(k).contiguous()
    vv = _bf16_bits(v).contiguous() if v is not None else None
    loc = _i64(cache_loc)
    n, hkv, lk = kk.shape
    lv = vv.shape[2] if vv is not None else 0
    lib.oracle_set_kv_buffer_fp8(
        _ptr(kk), *_row_strides(kk), _ptr(vv) if vv is not None else None,
        *(_row_strides(vv) if vv is not None else (0, 0)), _ptr(loc) if n else None, n, hkv,
        lk, lv, float(k_scale), float(v_scale), fmt, _ptr(kb), *_row_strides(kb), _ptr(vb),
        *_row_strides(vb))
    return kb.view(_FP8[fmt]), vb.view(_FP8[fmt])


def expand_paged_kv_indices(kv_indptr, kv_indices, kv_last_page_len, page_size, fill=-1):
    """Paged KV indices (sglang flashinfer_backend.py, the wrappers' paged
    format: indptr over pages, page indices, last_page_len, page_size) to
    per-token pool slots.  Returns (token_indptr int32 [bs+1], token_indices
    int32 [sum T_b]); ``fill`` marks entries not written."""
    lib = _load()
    kvp, kvi, lpl = _i32(kv_indptr), _i32(kv_indices), _i32(kv_last_page_len)
    bs = kvp.numel() - 1
    pages = (kvp[1:] - kvp[:-1]).to(torch.int64)
    t = torch.where(pages > 0, (pages - 1) * int(page_size) + lpl.to(torch.int64),
                    torch.zeros_like(pages))
    total = int(t.sum()) if bs else 0
    tptr = torch.empty(bs + 1, dtype=torch.int32)
    tidx = torch.full((total,), fill, dtype=torch.int32)
    lib.oracle_expand_paged_kv_indices(
        _ptr(kvp), _ptr(kvi) if kvi.numel() else None, _ptr(lpl) if bs else None,
        int(page_size), bs, _ptr(tptr), _ptr(tidx) if total else None)
    return tptr, tidx

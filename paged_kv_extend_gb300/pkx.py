"""Python binding of libpkx (include/pkx.h): argument marshalling only.

Every function here takes torch CUDA tensors, checks dtypes and shapes,
passes raw device pointers, element strides and the current CUDA stream to
the C entry point of the same name (``pkx_`` prefix dropped), and raises
:class:`PkxError` on a non-zero status.  All computation happens in the CUDA
kernels of libpkx.so; there is no fallback path.  If the library is missing
the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkx.so")

_p = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_f = ctypes.c_float
_sz = ctypes.c_size_t

_lock = threading.Lock()
_lib = None

# status codes (include/pkx.h)
PKX_OK, PKX_EINVAL, PKX_EUNSUPPORTED, PKX_ECUDA, PKX_ETIMEOUT, PKX_EDEVICE, PKX_EWORKSPACE = range(7)


class PkxError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"pkx error {code}: {msg}")
        self.code = code


# argtypes of every exported symbol, in header order
_SIGS = {
    "pkx_last_error_string": (ctypes.c_char_p, []),
    "pkx_version": (ctypes.c_char_p, []),
    "pkx_extend_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "pkx_decode_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "pkx_decode_workspace_min_size": (_sz, [_i, _i, _i, _i, _i]),
    "pkx_workspace_status": (_i, [_p, _p]),
    "pkx_set_attention_events": (None, [_p, _p]),
    "pkx_set_wait_limit_ns": (None, [ctypes.c_uint64]),
    "pkx_set_stall_injection": (None, [_i]),
    "pkx_extend_attention_fwd": (_i, [
        _p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i,
        _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _f, _f, _i, _p, _p, _p,
        _i, _f, _f, _p, _p, _sz, _p]),
    "pkx_extend_attention_fwd_kv_write": (_i, [
        _p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i,
        _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _f, _f, _i, _p, _p, _p,
        _i, _f, _f, _p, _p, _p, _sz, _p]),
    "pkx_ragged_paged_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "pkx_extend_attention_fwd_ragged_paged": (_i, [
        _p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i,
        _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _f, _f, _i, _i, _f, _f,
        _p, _p, _sz, _p]),
    "pkx_extend_attention_fwd_unified": (_i, [
        _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i,
        _i64, _i64, _i64, _i64, _i64, _f, _f, _i, _p, _p, _p, _i, _f, _f, _p, _p, _sz, _p]),
    "pkx_decode_attention_fwd": (_i, [
        _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i,
        _i64, _i64, _i64, _i64, _i64, _f, _f, _i, _i, _f, _f, _p, _p, _sz, _p]),
    "pkx_decode_attention_fwd_no_alloc": (_i, [
        _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i,
        _i64, _i64, _i64, _i64, _i64, _f, _f, _i, _p, _p]),
    "pkx_decode_no_alloc_status": (_i, [_p]),
    "pkx_merge_state": (_i, [_p, _p, _p, _p, _p, _p, _i64, _i, _i, _p]),
    "pkx_build_unified_kv_indices": (_i, [_p, _p, _p, _p, _p, _i, _p, _p, _p, _p]),
    "pkx_set_kv_buffer": (_i, [
        _p, _i64, _i64, _p, _i64, _i64, _p, _i64, _i, _i, _i,
        _p, _i64, _i64, _p, _i64, _i64, _i64, _p]),
    "pkx_set_kv_buffer_fp8": (_i, [
        _p, _i64, _i64, _p, _i64, _i64, _p, _i64, _i, _i, _i, _f, _f, _i,
        _p, _i64, _i64, _p, _i64, _i64, _i64, _p]),
    "pkx_expand_paged_kv_indices": (_i, [_p, _p, _p, _i, _i, _p, _p, _i64, _p]),
    "pkx_create_kv_indices": (_i, [
        _p, _i64, _i64, _p, _p, _p, _i, _p, _p, _i64, _p]),
}


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libpkx.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = path or LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libpkx.so not found at {path}: build it first "
                    "(python -m paged_kv_extend_gb300.build)")
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _check(rc: int):
    if rc != PKX_OK:
        msg = load_library().pkx_last_error_string().decode(errors="replace")
        raise PkxError(rc, msg)


def _ptr(t: Optional[torch.Tensor]):
    """Device address of ``t`` for a C entry point (every tensor argument of
    the library is a device pointer: a host tensor would reach a kernel as a
    host address, so it is refused here)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"expected a CUDA tensor, got one on {t.device} "
                         f"(shape {tuple(t.shape)}, {t.dtype})")
    return t.data_ptr()


def _on(dev: torch.device, fn, *args):
    """Call C entry point ``fn`` with ``dev`` as the calling thread's current
    CUDA device and that device's current stream as the last argument: the
    library launches on the current device, so a tensor on another GPU than
    the current one still gets its kernels on its own device."""
    with torch.cuda.device(dev):
        return fn(*args, torch.cuda.current_stream(dev).cuda_stream)


def _rows(t: torch.Tensor, name: str):
    if t.dim() != 3 or t.stride(2) != 1:
        raise ValueError(f"{name} must be [n, heads, dim] with a contiguous last dim")
    if t.dtype != torch.bfloat16 or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA bf16 tensor")
    return t.stride(0), t.stride(1)


# pool element formats (include/pkx.h PKX_KV_*)
PKX_KV_BF16, PKX_KV_FP8_E4M3, PKX_KV_FP8_E5M2 = 0, 1, 2
_KV_CODES = {torch.bfloat16: PKX_KV_BF16, torch.float8_e4m3fn: PKX_KV_FP8_E4M3,
             torch.float8_e5m2: PKX_KV_FP8_E5M2}


def _pool_rows(k_buffer: torch.Tensor, v_buffer: torch.Tensor):
    """Strides of a bf16 or fp8 pool pair and its PKX_KV_* format."""
    codes = [_KV_CODES.get(t.dtype) for t in (k_buffer, v_buffer)]
    if codes[0] is None or codes[0] != codes[1]:
        raise ValueError("k_buffer and v_buffer must both be bf16, float8_e4m3fn or float8_e5m2")
    out = []
    for t, nm in ((k_buffer, "k_buffer"), (v_buffer, "v_buffer")):
        if t.dim() != 3 or t.stride(2) != 1 or not t.is_cuda:
            raise ValueError(f"{nm} must be a CUDA [slots, heads, dim] tensor with a "
                             "contiguous last dim")
        out.append((t.stride(0), t.stride(1)))
    return out[0], out[1], codes[0]


def _i32(t: torch.Tensor, name: str):
    if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA int32 tensor")
    return t


def _mask_sinks(custom_mask, mask_indptr, sinks):
    """Check the optional custom mask (uint8, with int32 offsets) and sinks
    (fp32, one per query head) and return their pointers."""
    if custom_mask is not None:
        if custom_mask.dtype not in (torch.uint8, torch.bool) or not custom_mask.is_cuda or \
                not custom_mask.is_contiguous():
            raise ValueError("custom_mask must be a contiguous CUDA uint8/bool tensor")
        if mask_indptr is None:
            raise ValueError("custom_mask needs mask_indptr")
        _i32(mask_indptr, "mask_indptr")
    if sinks is not None and (sinks.dtype != torch.float32 or not sinks.is_cuda or
                              not sinks.is_contiguous()):
        raise ValueError("sinks must be a contiguous CUDA float32 tensor")
    return (_ptr(custom_mask), _ptr(mask_indptr) if custom_mask is not None else None,
            _ptr(sinks))


def version() -> str:
    return load_library().pkx_version().decode()


def extend_workspace_size(batch, num_q_tokens, hq, hkv, lq, lv) -> int:
    return int(load_library().pkx_extend_workspace_size(batch, num_q_tokens, hq, hkv, lq, lv))


def decode_workspace_size(batch, hq, hkv, lq, lv) -> int:
    return int(load_library().pkx_decode_workspace_size(batch, hq, hkv, lq, lv))


def decode_workspace_min_size(batch, hq, hkv, lq, lv) -> int:
    """The smallest decode workspace (one key stream per unit)."""
    return int(load_library().pkx_decode_workspace_min_size(batch, hq, hkv, lq, lv))


def workspace_status(workspace: torch.Tensor) -> int:
    """Status word of the last attention call that used ``workspace``
    (synchronises the current stream).  Returns the code; does not raise."""
    return int(_on(workspace.device, load_library().pkx_workspace_status, _ptr(workspace)))


def set_attention_events(before=None, after=None):
    """Record CUDA events ``before``/``after`` (torch.cuda.Event, already
    recorded once so that they exist) around the attention kernel of every
    later attention call on this thread; ``None, None`` stops."""
    load_library().pkx_set_attention_events(
        None if before is None else before.cuda_event,
        None if after is None else after.cuda_event)


def set_wait_limit_ns(ns: int = 0):
    """Time limit (ns) of the bounded device waits of attention kernels
    launched later on this thread; 0 restores the default (two seconds)."""
    load_library().pkx_set_wait_limit_ns(int(ns))


def set_stall_injection(on: bool):
    """Test hook: while on, attention kernels launched on this thread stall
    their softmax warps on a barrier nothing arrives at, so the bounded wait
    runs out and the call reports PKX_ETIMEOUT."""
    load_library().pkx_set_stall_injection(1 if on else 0)


def _check_attn(q, o, lse, k_buffer, v_buffer, n_q, hq, lq, lv):
    """Host-side shape checks of an attention call (the C entry points take
    raw pointers, so an undersized output would be written out of bounds)."""
    for t, nm in ((q, "q"), (o, "o")):
        if t.dim() != 3 or not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError(f"{nm} must be a contiguous bf16 [tokens, heads, dim] tensor")
    if tuple(o.shape) != (n_q, hq, lv):
        raise ValueError(f"o has shape {tuple(o.shape)}, expected {(n_q, hq, lv)}")
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous() or
                            tuple(lse.shape) != (n_q, hq)):
        raise ValueError(f"lse must be a contiguous float32 [{n_q}, {hq}] tensor")
    if (k_buffer.dim() != 3 or v_buffer.dim() != 3 or k_buffer.shape[0] != v_buffer.shape[0]
            or k_buffer.shape[1] != v_buffer.shape[1] or k_buffer.shape[2] != lq):
        raise ValueError("k_buffer [slots, Hkv, Lq] and v_buffer [slots, Hkv, Lv] disagree "
                         f"with each other or with q's Lq={lq}")


def _check_len(t, n, name):
    if t.numel() != n:
        raise ValueError(f"{name} has {t.numel()} entries, expected {n}")


def _workspace(ws, nbytes, dev):
    """The caller's workspace (its size is checked by the library), or a new
    one of the size the library asks for."""
    if ws is None:
        return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    return ws


def extend_attention_fwd(q_extend, k_extend, v_extend, o_extend, k_buffer, v_buffer,
                         qo_indptr, kv_indptr, kv_indices, sm_scale=None, logit_cap=0.0,
                         sliding_window=-1, lse=None, workspace=None, custom_mask=None,
                         mask_indptr=None, sinks=None, k_scale=1.0, v_scale=1.0,
                         cache_loc=None):
    """Two-stage extend attention (pkx_extend_attention_fwd); writes o_extend
    (and lse if given) in place.  Returns the workspace used.  custom_mask /
    mask_indptr / sinks as in the C header.  The pool may be fp8
    (torch.float8_e4m3fn / float8_e5m2) with k_scale / v_scale.  With
    ``cache_loc`` (int64 [tokens], each extend token's pool slot) the call
    also stores k_extend / v_extend into the pool at those slots
    (pkx_extend_attention_fwd_kv_write)."""
    lib = load_library()
    n, hq, lq = q_extend.shape
    hkv = k_buffer.shape[1]
    lv = v_buffer.shape[2]
    batch = qo_indptr.numel() - 1
    _check_attn(q_extend, o_extend, lse, k_buffer, v_buffer, n, hq, lq, lv)
    _check_len(kv_indptr, batch + 1, "kv_indptr")
    if tuple(k_extend.shape) != (n, hkv, lq) or tuple(v_extend.shape) != (n, hkv, lv):
        raise ValueError("k_extend / v_extend must be [tokens, Hkv, Lq] / [tokens, Hkv, Lv] "
                         "with q's token count")
    ke = _rows(k_extend, "k_extend")
    ve = _rows(v_extend, "v_extend")
    kb, vb, kv_dtype = _pool_rows(k_buffer, v_buffer)
    for t, nm in ((q_extend, "q_extend"), (o_extend, "o_extend")):
        if not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError(f"{nm} must be contiguous bf16")
    _i32(qo_indptr, "qo_indptr"), _i32(kv_indptr, "kv_indptr"), _i32(kv_indices, "kv_indices")
    ws = _workspace(workspace, extend_workspace_size(batch, n, hq, hkv, lq, lv), q_extend.device)
    args = [
        _ptr(q_extend), _ptr(k_extend), _ptr(v_extend), _ptr(o_extend), _ptr(k_buffer),
        _ptr(v_buffer), _ptr(qo_indptr), _ptr(kv_indptr),
        _ptr(kv_indices) if kv_indices.numel() else None, batch, n, hq, hkv, lq, lv,
        ke[0], ke[1], ve[0], ve[1], kb[0], kb[1], vb[0], vb[1], k_buffer.shape[0],
        float(sm_scale or 0.0), float(logit_cap or 0.0), int(sliding_window),
        *_mask_sinks(custom_mask, mask_indptr, sinks), kv_dtype, float(k_scale), float(v_scale),
        _ptr(lse)]
    if cache_loc is None:
        _check(_on(q_extend.device, lib.pkx_extend_attention_fwd, *args, _ptr(ws),
                   ws.numel() * ws.element_size()))
    else:
        _i64_vec(cache_loc, "cache_loc")
        _check_len(cache_loc, n, "cache_loc")
        _check(_on(q_extend.device, lib.pkx_extend_attention_fwd_kv_write, *args,
                   _ptr(cache_loc) if n else None, _ptr(ws), ws.numel() * ws.element_size()))
    return ws


def ragged_paged_workspace_size(batch, num_q_tokens, hq, hkv, lq, lv) -> int:
    return int(load_library().pkx_ragged_paged_workspace_size(batch, num_q_tokens, hq, hkv,
                                                               lq, lv))


def extend_attention_fwd_ragged_paged(q_extend, k_extend, v_extend, o_extend, k_buffer,
                                      v_buffer, qo_indptr, kv_indptr, kv_indices, sm_scale=None,
                                      logit_cap=0.0, sliding_window=-1, lse=None,
                                      workspace=None, k_scale=1.0, v_scale=1.0):
    """Extend attention as a ragged pass over the extend keys, a paged pass
    over the prefix keys and merge_state of the two
    (pkx_extend_attention_fwd_ragged_paged); arguments as
    extend_attention_fwd without mask and sinks.  Returns the workspace."""
    lib = load_library()
    n, hq, lq = q_extend.shape
    hkv = k_buffer.shape[1]
    lv = v_buffer.shape[2]
    batch = qo_indptr.numel() - 1
    _check_attn(q_extend, o_extend, lse, k_buffer, v_buffer, n, hq, lq, lv)
    _check_len(kv_indptr, batch + 1, "kv_indptr")
    if tuple(k_extend.shape) != (n, hkv, lq) or tuple(v_extend.shape) != (n, hkv, lv):
        raise ValueError("k_extend / v_extend must be [tokens, Hkv, Lq] / [tokens, Hkv, Lv] "
                         "with q's token count")
    ke = _rows(k_extend, "k_extend")
    ve = _rows(v_extend, "v_extend")
    kb, vb, kv_dtype = _pool_rows(k_buffer, v_buffer)
    for t, nm in ((q_extend, "q_extend"), (o_extend, "o_extend")):
        if not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError(f"{nm} must be contiguous bf16")
    _i32(qo_indptr, "qo_indptr"), _i32(kv_indptr, "kv_indptr"), _i32(kv_indices, "kv_indices")
    ws = _workspace(workspace, ragged_paged_workspace_size(batch, n, hq, hkv, lq, lv),
                    q_extend.device)
    _check(_on(
        q_extend.device, lib.pkx_extend_attention_fwd_ragged_paged,
        _ptr(q_extend), _ptr(k_extend), _ptr(v_extend), _ptr(o_extend), _ptr(k_buffer),
        _ptr(v_buffer), _ptr(qo_indptr), _ptr(kv_indptr),
        _ptr(kv_indices) if kv_indices.numel() else None, batch, n, hq, hkv, lq, lv,
        ke[0], ke[1], ve[0], ve[1], kb[0], kb[1], vb[0], vb[1], k_buffer.shape[0],
        float(sm_scale or 0.0), float(logit_cap or 0.0), int(sliding_window), kv_dtype,
        float(k_scale), float(v_scale), _ptr(lse), _ptr(ws), ws.numel() * ws.element_size()))
    return ws


def extend_attention_fwd_unified(q, o, k_buffer, v_buffer, qo_indptr, kv_indptr, kv_indices,
                                 prefix_lens, sm_scale=None, logit_cap=0.0, sliding_window=-1,
                                 lse=None, workspace=None, custom_mask=None, mask_indptr=None,
                                 sinks=None, k_scale=1.0, v_scale=1.0):
    """Unified extend attention (pkx_extend_attention_fwd_unified); int64
    kv_indices over every key.  Writes o (and lse) in place.  The pool may be
    fp8 (torch.float8_e4m3fn / float8_e5m2) with k_scale / v_scale."""
    lib = load_library()
    n, hq, lq = q.shape
    hkv = k_buffer.shape[1]
    lv = v_buffer.shape[2]
    batch = qo_indptr.numel() - 1
    _check_attn(q, o, lse, k_buffer, v_buffer, n, hq, lq, lv)
    _check_len(kv_indptr, batch + 1, "kv_indptr")
    _check_len(prefix_lens, batch, "prefix_lens")
    kb, vb, kv_dtype = _pool_rows(k_buffer, v_buffer)
    if kv_indices.dtype != torch.int64 or not kv_indices.is_contiguous():
        raise ValueError("kv_indices must be contiguous int64")
    _i32(qo_indptr, "qo_indptr"), _i32(kv_indptr, "kv_indptr"), _i32(prefix_lens, "prefix_lens")
    ws = _workspace(workspace, extend_workspace_size(batch, n, hq, hkv, lq, lv), q.device)
    _check(_on(
        q.device, lib.pkx_extend_attention_fwd_unified,
        _ptr(q), _ptr(o), _ptr(k_buffer), _ptr(v_buffer), _ptr(qo_indptr), _ptr(kv_indptr),
        _ptr(kv_indices) if kv_indices.numel() else None, _ptr(prefix_lens), batch, n, hq, hkv,
        lq, lv, kb[0], kb[1], vb[0], vb[1], k_buffer.shape[0], float(sm_scale or 0.0),
        float(logit_cap or 0.0), int(sliding_window),
        *_mask_sinks(custom_mask, mask_indptr, sinks), kv_dtype, float(k_scale),
        float(v_scale), _ptr(lse), _ptr(ws), ws.numel() * ws.element_size()))
    return ws


def decode_attention_fwd(q, o, k_buffer, v_buffer, kv_indptr, kv_indices, sm_scale=None,
                         logit_cap=0.0, sliding_window=-1, lse=None, workspace=None,
                         k_scale=1.0, v_scale=1.0):
    """Decode attention (pkx_decode_attention_fwd): q [B, Hq, Lq] -> o.  The
    pool may be fp8 (torch.float8_e4m3fn / float8_e5m2) with k_scale /
    v_scale.  A given ``workspace`` of at least decode_workspace_min_size
    bytes is accepted (two key streams per unit from decode_workspace_size
    bytes up, one below)."""
    lib = load_library()
    b, hq, lq = q.shape
    hkv = k_buffer.shape[1]
    lv = v_buffer.shape[2]
    _check_attn(q, o, lse, k_buffer, v_buffer, b, hq, lq, lv)
    _check_len(kv_indptr, b + 1, "kv_indptr")
    kb, vb, kv_dtype = _pool_rows(k_buffer, v_buffer)
    _i32(kv_indptr, "kv_indptr"), _i32(kv_indices, "kv_indices")
    ws = _workspace(workspace, decode_workspace_size(b, hq, hkv, lq, lv), q.device)
    _check(_on(
        q.device, lib.pkx_decode_attention_fwd,
        _ptr(q), _ptr(o), _ptr(k_buffer), _ptr(v_buffer), _ptr(kv_indptr),
        _ptr(kv_indices) if kv_indices.numel() else None, b, hq, hkv, lq, lv,
        kb[0], kb[1], vb[0], vb[1], k_buffer.shape[0], float(sm_scale or 0.0),
        float(logit_cap or 0.0), int(sliding_window), kv_dtype, float(k_scale),
        float(v_scale), _ptr(lse), _ptr(ws),
        ws.numel() * ws.element_size()))
    return ws


def decode_attention_fwd_no_alloc(q, o, k_buffer, v_buffer, kv_indptr, kv_indices,
                                  sm_scale=None, logit_cap=0.0, sliding_window=-1, lse=None):
    """Decode attention with the library's built-in scratch instead of a
    workspace (pkx_decode_attention_fwd_no_alloc), for callers that cannot
    allocate device memory.  Calls that overlap on the GPU must not be made."""
    lib = load_library()
    b, hq, lq = q.shape
    hkv = k_buffer.shape[1]
    lv = v_buffer.shape[2]
    _check_attn(q, o, lse, k_buffer, v_buffer, b, hq, lq, lv)
    _check_len(kv_indptr, b + 1, "kv_indptr")
    kb = _rows(k_buffer, "k_buffer")
    vb = _rows(v_buffer, "v_buffer")
    _i32(kv_indptr, "kv_indptr"), _i32(kv_indices, "kv_indices")
    _check(_on(
        q.device, lib.pkx_decode_attention_fwd_no_alloc,
        _ptr(q), _ptr(o), _ptr(k_buffer), _ptr(v_buffer), _ptr(kv_indptr),
        _ptr(kv_indices) if kv_indices.numel() else None, b, hq, hkv, lq, lv,
        kb[0], kb[1], vb[0], vb[1], k_buffer.shape[0], float(sm_scale or 0.0),
        float(logit_cap or 0.0), int(sliding_window), _ptr(lse)))


def decode_no_alloc_status(device=None) -> int:
    """Status word of the last allocation-free decode call on ``device``
    (default: the current one), read back like workspace_status (synchronises
    that device's current stream).  Returns the code; does not raise."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else \
        torch.device(device)
    return int(_on(dev, load_library().pkx_decode_no_alloc_status))


def merge_state(v_a, s_a, v_b, s_b, v_out=None, s_out=None):
    """merge_state (pkx_merge_state).  Returns (v_out, s_out)."""
    lib = load_library()
    n, h, dv = v_a.shape
    if v_out is None:
        v_out = torch.empty_like(v_a)
    if s_out is None:
        s_out = torch.empty_like(s_a)
    for t in (v_a, v_b, v_out):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or t.shape != v_a.shape:
            raise ValueError("v tensors must be contiguous bf16 of v_a's shape")
    for t in (s_a, s_b, s_out):
        if t.dtype != torch.float32 or not t.is_contiguous() or tuple(t.shape) != (n, h):
            raise ValueError(f"s tensors must be contiguous fp32 [{n}, {h}]")
    _check(_on(v_a.device, lib.pkx_merge_state, _ptr(v_a), _ptr(s_a), _ptr(v_b), _ptr(s_b),
               _ptr(v_out), _ptr(s_out), n, h, dv))
    return v_out, s_out


def build_unified_kv_indices(prefix_kv_indptr, prefix_kv_indices, extend_start_loc,
                             extend_seq_lens, extend_kv_indices, bs, out=None):
    """Unified KV-index build (pkx_build_unified_kv_indices).  Returns
    (unified_kv_indptr int32 [bs+1], unified_kv_indices int64, prefix_lens
    int32 [bs]); pass ``out`` = that triple to write into existing tensors."""
    lib = load_library()
    dev = prefix_kv_indptr.device
    for t, nm in ((prefix_kv_indptr, "prefix_kv_indptr"), (prefix_kv_indices, "prefix_kv_indices"),
                  (extend_start_loc, "extend_start_loc"), (extend_seq_lens, "extend_seq_lens"),
                  (extend_kv_indices, "extend_kv_indices")):
        _i32(t, nm)
    _check_len(prefix_kv_indptr, bs + 1, "prefix_kv_indptr")
    _check_len(extend_start_loc, bs, "extend_start_loc")
    _check_len(extend_seq_lens, bs, "extend_seq_lens")
    n_idx = prefix_kv_indices.numel() + extend_kv_indices.numel()
    if out is None:
        uptr = torch.empty(bs + 1, dtype=torch.int32, device=dev)
        uidx = torch.empty(n_idx, dtype=torch.int64, device=dev)
        plen = torch.empty(bs, dtype=torch.int32, device=dev)
    else:
        uptr, uidx, plen = out
        _i32(uptr, "unified_kv_indptr"), _i32(plen, "prefix_lens")
        _check_len(uptr, bs + 1, "unified_kv_indptr")
        _check_len(plen, bs, "prefix_lens")
        if uidx.dtype != torch.int64 or not uidx.is_contiguous() or uidx.device != dev:
            raise ValueError("unified_kv_indices must be a contiguous int64 tensor on "
                             f"{dev}")
        if uidx.numel() < n_idx:
            raise ValueError(f"unified_kv_indices holds {uidx.numel()} entries, fewer than the "
                             f"{n_idx} prefix + extend indices")
    for t, nm in ((uptr, "unified_kv_indptr"), (plen, "prefix_lens")):
        if t.device != dev:
            raise ValueError(f"{nm} must be on {dev}")
    _check(_on(
        dev, lib.pkx_build_unified_kv_indices,
        _ptr(prefix_kv_indptr), _ptr(prefix_kv_indices) if prefix_kv_indices.numel() else None,
        _ptr(extend_start_loc), _ptr(extend_seq_lens),
        _ptr(extend_kv_indices) if extend_kv_indices.numel() else None, int(bs), _ptr(uptr),
        _ptr(uidx) if uidx.numel() else None, _ptr(plen)))
    return uptr, uidx, plen


def _i64_vec(t: torch.Tensor, name: str):
    if t.dtype != torch.int64 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA int64 tensor")
    return t


def set_kv_buffer(k_buffer, v_buffer, cache_loc, k, v=None):
    """KV write into the pool (pkx_set_kv_buffer): row cache_loc[t] of every
    KV head of k_buffer / v_buffer becomes k[t] / v[t], in place.  ``v`` None
    writes K only (a K-only MLA pool).  cache_loc int64 [n]."""
    lib = load_library()
    _i64_vec(cache_loc, "cache_loc")
    n, hkv, lk = k.shape
    if cache_loc.numel() != n:
        raise ValueError("cache_loc must hold one slot per token")
    ks, kbs = _rows(k, "k"), _rows(k_buffer, "k_buffer")
    if k_buffer.shape[1] != hkv or k_buffer.shape[2] != lk:
        raise ValueError("k_buffer must be [slots, hkv, lk] like k")
    lv, vs, vbs = 0, (0, 0), (0, 0)
    if v is not None:
        vs, vbs = _rows(v, "v"), _rows(v_buffer, "v_buffer")
        lv = v.shape[2]
        if v.shape[:2] != (n, hkv) or v_buffer.shape[1:] != (hkv, lv):
            raise ValueError("v / v_buffer shapes do not match k")
        if v_buffer.shape[0] != k_buffer.shape[0]:
            raise ValueError("k_buffer and v_buffer must have the same number of slots")
    _check(_on(
        k.device, lib.pkx_set_kv_buffer,
        _ptr(k), ks[0], ks[1], _ptr(v), vs[0], vs[1], _ptr(cache_loc) if n else None, n, hkv,
        lk, lv, _ptr(k_buffer), kbs[0], kbs[1], _ptr(v_buffer) if v is not None else None,
        vbs[0], vbs[1], k_buffer.shape[0]))
    return k_buffer, v_buffer


def create_kv_indices(req_to_token, req_pool_indices, paged_kernel_lens, kv_start_idx=None,
                      kv_indptr=None, kv_indices=None, capacity=None):
    """KV-index gather from the request-to-token table
    (pkx_create_kv_indices).  req_to_token int32 [rows, cols];
    req_pool_indices, paged_kernel_lens, kv_start_idx int64 [bs].  Returns
    (kv_indptr int32 [bs+1], kv_indices int32).  Without ``kv_indices`` the
    output is allocated with ``capacity`` entries, which the caller must
    give (the host knows the sum of paged_kernel_lens; reading it back here
    would synchronise)."""
    lib = load_library()
    if req_to_token.dtype != torch.int32 or not req_to_token.is_cuda or \
            req_to_token.dim() != 2 or not req_to_token.is_contiguous():
        raise ValueError("req_to_token must be a contiguous CUDA int32 [rows, cols] tensor")
    _i64_vec(req_pool_indices, "req_pool_indices")
    _i64_vec(paged_kernel_lens, "paged_kernel_lens")
    if kv_start_idx is not None:
        _i64_vec(kv_start_idx, "kv_start_idx")
    bs = req_pool_indices.numel()
    dev = req_to_token.device
    if kv_indptr is None:
        kv_indptr = torch.empty(bs + 1, dtype=torch.int32, device=dev)
    if kv_indices is None:
        if capacity is None:
            raise ValueError("give kv_indices or capacity (the sum of paged_kernel_lens)")
        kv_indices = torch.empty(int(capacity), dtype=torch.int32, device=dev)
    _i32(kv_indptr, "kv_indptr")
    _i32(kv_indices, "kv_indices")
    _check(_on(
        dev, lib.pkx_create_kv_indices,
        _ptr(req_to_token) if req_to_token.numel() else None, req_to_token.shape[0],
        req_to_token.stride(0), _ptr(req_pool_indices) if bs else None,
        _ptr(paged_kernel_lens) if bs else None,
        _ptr(kv_start_idx) if kv_start_idx is not None and bs else None, int(bs),
        _ptr(kv_indptr), _ptr(kv_indices) if kv_indices.numel() else None,
        kv_indices.numel()))
    return kv_indptr, kv_indices


def set_kv_buffer_fp8(k_buffer, v_buffer, cache_loc, k, v, k_scale, v_scale):
    """KV write into an fp8 pool (pkx_set_kv_buffer_fp8): k[t] / k_scale and
    v[t] / v_scale as fp8 codes at slot cache_loc[t], in place.  Pools are
    torch.float8_e4m3fn or float8_e5m2 [slots, hkv, d]; ``v`` None writes K
    only."""
    lib = load_library()
    _i64_vec(cache_loc, "cache_loc")
    n, hkv, lk = k.shape
    if cache_loc.numel() != n:
        raise ValueError("cache_loc must hold one slot per token")
    kb, vb, fmt = _pool_rows(k_buffer, v_buffer)
    if fmt == PKX_KV_BF16:
        raise ValueError("set_kv_buffer_fp8 needs fp8 pools")
    ks = _rows(k, "k")
    lv, vs = 0, (0, 0)
    if v is not None:
        vs = _rows(v, "v")
        lv = v.shape[2]
    _check(_on(
        k.device, lib.pkx_set_kv_buffer_fp8,
        _ptr(k), ks[0], ks[1], _ptr(v), vs[0], vs[1], _ptr(cache_loc) if n else None, n, hkv,
        lk, lv, float(k_scale), float(v_scale), fmt, _ptr(k_buffer), kb[0], kb[1],
        _ptr(v_buffer) if v is not None else None, vb[0], vb[1], k_buffer.shape[0]))
    return k_buffer, v_buffer


def expand_paged_kv_indices(kv_indptr, kv_indices, kv_last_page_len, page_size,
                            token_indptr=None, token_indices=None, capacity=None):
    """Paged KV indices (page size > 1) to per-token pool slots
    (pkx_expand_paged_kv_indices).  All int32 CUDA tensors.  Returns
    (token_indptr [bs+1], token_indices); without ``token_indices`` the output
    is allocated with ``capacity`` entries (the host-known key count)."""
    lib = load_library()
    for t, nm in ((kv_indptr, "kv_indptr"), (kv_indices, "kv_indices"),
                  (kv_last_page_len, "kv_last_page_len")):
        _i32(t, nm)
    bs = kv_indptr.numel() - 1
    dev = kv_indptr.device
    if token_indptr is None:
        token_indptr = torch.empty(bs + 1, dtype=torch.int32, device=dev)
    if token_indices is None:
        if capacity is None:
            raise ValueError("give token_indices or capacity (the total key count)")
        token_indices = torch.empty(int(capacity), dtype=torch.int32, device=dev)
    _i32(token_indptr, "token_indptr")
    _i32(token_indices, "token_indices")
    _check(_on(
        dev, lib.pkx_expand_paged_kv_indices,
        _ptr(kv_indptr), _ptr(kv_indices) if kv_indices.numel() else None,
        _ptr(kv_last_page_len), int(page_size), int(bs), _ptr(token_indptr),
        _ptr(token_indices) if token_indices.numel() else None, token_indices.numel()))
    return token_indptr, token_indices

"""ctypes binding of libattn_sink.so (argument marshalling only).

Every step of the computation runs in the library's CUDA kernels; this module
only checks tensor dtypes/devices, allocates outputs with torch and passes raw
pointers, sizes and the current CUDA stream through the C ABI.  There is no
fallback: if the shared library is missing the import fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn_sink.so")

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE = 0, -1, -2, -3, -4
DEV_PAGE_OOB, DEV_SEQLEN_OOB, DEV_TIMEOUT, DEV_LAYOUT = 1, 2, 4, 8

_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_longlong
_F = ctypes.c_float

_SIGS = {
    "attn_sink_fwd": [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P,
                      _P],
    "attn_sink_decode_paged": [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P, _I, _I, _F, _P, _P, _P],
    "attn_sink_decode_paged_noalloc": [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P, _I, _I, _F, _P,
                                       _P, _P],
    "attn_sink_bwd": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                      _I, _F, _P, _P, _P, _P, _P],
    "attn_sink_fwd_host": [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P],
    "attn_sink_fwd_strided": [_P, _P, _P, _L, _L, _L, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                              _I, _F, _P, _P, _P],
    "attn_sink_bwd_strided": [_P, _P, _P, _L, _L, _L, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                              _I, _I, _I, _I, _F, _P, _P, _P, _L, _L, _L, _P, _P],
    "attn_sink_kv_append": [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P],
    "attn_sink_decode_paged_append": [_P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P, _I, _I, _F,
                                      _P, _P, _P],
    "attn_sink_fwd_paged": [_P, _P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _I,
                            _I, _I, _F, _P, _P, _P],
    "attn_sink_visible_ranges": [_P, _I, _I, _I, _P, _P],
    "attn_sink_visible_slots": [_P, _P, _I, _I, _I, _I, _I, _I, _P, _I, _P],
    "attn_sink_device_status": [_P],
    "attn_sink_selftest_wait": [_I, _P],
    "attn_sink_last_error": [],
    "attn_sink_version": [],
}

EXPORTS = tuple(_SIGS)


class AttnSinkError(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__(f"{fn} returned {code}: {msg}")
        self.code = code


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it first (python -m paged_kv_sink_gb300.build)")
    lib = ctypes.CDLL(path)
    for name, args in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_char_p if name in ("attn_sink_last_error", "attn_sink_version") else ctypes.c_int
    return lib


_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load()
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(name, rc):
    if rc != OK:
        msg = lib().attn_sink_last_error().decode()
        raise AttnSinkError(name, rc, msg)


def _need(t, dtype, name, dev=True):
    if t is None:
        return
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if dev and not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise TypeError(f"{name} must be contiguous")


def attn_sink_fwd(q, k, v, sink, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                  win_first=0, win_last=0, causal=True, scale=0.0, out=None, lse=None,
                  return_lse=True, stream=None):
    """Varlen forward with a sink.  q (Tq,Hq,d), k/v (Tk,Hkv,d) bf16 CUDA; returns (out, lse)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    _need(sink, torch.float32, "sink")
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q")
    _need(cu_seqlens_k, torch.int32, "cu_seqlens_k")
    tq, hq, d = q.shape
    hkv = k.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((hq, tq), dtype=torch.float32, device=q.device)
    rc = lib().attn_sink_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(sink), _ptr(cu_seqlens_q),
                             _ptr(cu_seqlens_k), cu_seqlens_q.numel() - 1, tq, k.shape[0], hq, hkv,
                             d, int(max_seqlen_q), int(max_seqlen_k), int(win_first), int(win_last),
                             1 if causal else 0, float(scale), _ptr(out), _ptr(lse), _stream(stream))
    _check("attn_sink_fwd", rc)
    return out, lse


def attn_sink_fwd_host(q, k, v, sink, cu_seqlens_q, cu_seqlens_k, win_first=0, win_last=0, causal=True,
                       scale=0.0, out=None, lse=None, return_lse=True, stream=None):
    """attn_sink_fwd on host (CPU, preferably pinned) tensors: the library moves
    each request's rows to the device and back, pipelined against the kernels.
    Returns (out, lse) as host tensors; they are valid after ``stream`` (default:
    the current CUDA stream) is synchronised."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n, dev=False)
    _need(sink, torch.float32, "sink", dev=False)
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q", dev=False)
    _need(cu_seqlens_k, torch.int32, "cu_seqlens_k", dev=False)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (sink, "sink"), (cu_seqlens_q, "cu_seqlens_q"),
                 (cu_seqlens_k, "cu_seqlens_k")):
        if t is not None and t.is_cuda:
            raise TypeError(f"{n} must be a host tensor")
    tq, hq, d = q.shape
    hkv = k.shape[1]
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    if lse is None and return_lse:
        lse = torch.empty((hq, tq), dtype=torch.float32, pin_memory=True)
    rc = lib().attn_sink_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(sink), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                                  cu_seqlens_q.numel() - 1, hq, hkv, d, int(win_first), int(win_last),
                                  1 if causal else 0, float(scale), _ptr(out), _ptr(lse), _stream(stream))
    _check("attn_sink_fwd_host", rc)
    return out, lse


def attn_sink_decode_paged(q, k_cache, v_cache, page_table, seqlens, sink=None, win_first=0,
                           win_last=0, scale=0.0, out=None, lse=None, return_lse=True, stream=None,
                           _entry="attn_sink_decode_paged"):
    """Paged decode.  q (B,Hq,d); caches (P,ps,Hkv,d); page_table (B,maxp) int32; seqlens (B,)."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n)
    _need(page_table, torch.int32, "page_table")
    _need(seqlens, torch.int32, "seqlens")
    _need(sink, torch.float32, "sink")
    B, hq, d = q.shape
    npages, ps, hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, hq), dtype=torch.float32, device=q.device)
    rc = getattr(lib(), _entry)(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table),
                                page_table.shape[1], _ptr(seqlens), B, hq, hkv, d, ps, npages,
                                _ptr(sink), int(win_first), int(win_last), float(scale),
                                _ptr(out), _ptr(lse), _stream(stream))
    _check(_entry, rc)
    return out, lse


def attn_sink_decode_paged_noalloc(q, k_cache, v_cache, page_table, seqlens, sink=None, win_first=0,
                                   win_last=0, scale=0.0, out=None, lse=None, return_lse=True,
                                   stream=None):
    """Allocation-free paged decode: the library allocates no device memory
    for the call (its scratch is a static device array).  Outputs are still
    allocated here by torch unless ``out``/``lse`` are given."""
    return attn_sink_decode_paged(q, k_cache, v_cache, page_table, seqlens, sink, win_first, win_last,
                                  scale, out, lse, return_lse, stream,
                                  _entry="attn_sink_decode_paged_noalloc")


def _row_view(base, col0, heads, d):
    """(pointer, row stride) of columns [col0, col0 + heads) of a (T, C, d) buffer."""
    if base.dim() != 3 or base.stride(2) != 1 or base.stride(1) != d:
        raise TypeError("packed buffer must be (T, C, d) with contiguous rows")
    return ctypes.c_void_p(base.data_ptr() + col0 * d * base.element_size()), base.stride(0)


def attn_sink_fwd_qkvpacked(qkv, hkv, sink, cu_seqlens_q, max_seqlen_q, win_first=0, win_last=0,
                            causal=True, scale=0.0, out=None, lse=None, return_lse=True, stream=None):
    """Self-attention forward on a packed (T, hq + 2*hkv, d) QKV buffer (a
    (T, 3, H, d) buffer is the same with hkv = H after a view).  Returns (out, lse)."""
    if qkv.dim() == 4:
        qkv = qkv.reshape(qkv.shape[0], -1, qkv.shape[-1])
    _need(qkv, torch.bfloat16, "qkv")
    _need(sink, torch.float32, "sink")
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q")
    T, C, d = qkv.shape
    hq = C - 2 * hkv
    qp, rs = _row_view(qkv, 0, hq, d)
    kp, _ = _row_view(qkv, hq, hkv, d)
    vp, _ = _row_view(qkv, hq + hkv, hkv, d)
    if out is None:
        out = torch.empty((T, hq, d), dtype=qkv.dtype, device=qkv.device)
    if lse is None and return_lse:
        lse = torch.empty((hq, T), dtype=torch.float32, device=qkv.device)
    rc = lib().attn_sink_fwd_strided(qp, kp, vp, rs, rs, rs, _ptr(sink), _ptr(cu_seqlens_q), _ptr(cu_seqlens_q),
                                     cu_seqlens_q.numel() - 1, T, T, hq, hkv, d, int(max_seqlen_q),
                                     int(max_seqlen_q), int(win_first), int(win_last), 1 if causal else 0,
                                     float(scale), _ptr(out), _ptr(lse), _stream(stream))
    _check("attn_sink_fwd_strided", rc)
    return out, lse


def attn_sink_fwd_kvpacked(q, kv, sink, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, win_first=0,
                           win_last=0, causal=True, scale=0.0, out=None, lse=None, return_lse=True,
                           stream=None):
    """Forward with a packed (Tk, 2, hkv, d) KV buffer.  Returns (out, lse)."""
    _need(q, torch.bfloat16, "q")
    _need(kv, torch.bfloat16, "kv")
    _need(sink, torch.float32, "sink")
    tq, hq, d = q.shape
    tk, _, hkv, _ = kv.shape
    kv3 = kv.reshape(tk, 2 * hkv, d)
    kp, rs = _row_view(kv3, 0, hkv, d)
    vp, _ = _row_view(kv3, hkv, hkv, d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((hq, tq), dtype=torch.float32, device=q.device)
    rc = lib().attn_sink_fwd_strided(_ptr(q), kp, vp, 0, rs, rs, _ptr(sink), _ptr(cu_seqlens_q),
                                     _ptr(cu_seqlens_k), cu_seqlens_q.numel() - 1, tq, tk, hq, hkv, d,
                                     int(max_seqlen_q), int(max_seqlen_k), int(win_first), int(win_last),
                                     1 if causal else 0, float(scale), _ptr(out), _ptr(lse), _stream(stream))
    _check("attn_sink_fwd_strided", rc)
    return out, lse


def attn_sink_bwd_qkvpacked(qkv, hkv, sink, out, lse, dout, cu_seqlens_q, max_seqlen_q, win_first=0,
                            win_last=0, causal=True, scale=0.0, dqkv=None, dsink=None, stream=None):
    """Backward of attn_sink_fwd_qkvpacked; returns (dqkv, dsink or None), dqkv in
    the layout of qkv."""
    shape4 = qkv.shape if qkv.dim() == 4 else None
    if qkv.dim() == 4:
        qkv = qkv.reshape(qkv.shape[0], -1, qkv.shape[-1])
    for t, n in ((qkv, "qkv"), (out, "out"), (dout, "dout")):
        _need(t, torch.bfloat16, n)
    _need(sink, torch.float32, "sink")
    _need(lse, torch.float32, "lse")
    T, C, d = qkv.shape
    hq = C - 2 * hkv
    dqkv = torch.empty_like(qkv) if dqkv is None else dqkv.reshape(T, C, d)
    if sink is not None and dsink is None:
        dsink = torch.empty_like(sink)
    qp, rs = _row_view(qkv, 0, hq, d)
    kp, _ = _row_view(qkv, hq, hkv, d)
    vp, _ = _row_view(qkv, hq + hkv, hkv, d)
    dqp, drs = _row_view(dqkv, 0, hq, d)
    dkp, _ = _row_view(dqkv, hq, hkv, d)
    dvp, _ = _row_view(dqkv, hq + hkv, hkv, d)
    rc = lib().attn_sink_bwd_strided(qp, kp, vp, rs, rs, rs, _ptr(sink), _ptr(out), _ptr(lse), _ptr(dout),
                                     _ptr(cu_seqlens_q), _ptr(cu_seqlens_q), cu_seqlens_q.numel() - 1, T, T, hq,
                                     hkv, d, int(max_seqlen_q), int(max_seqlen_q), int(win_first),
                                     int(win_last), 1 if causal else 0, float(scale), dqp, dkp, dvp, drs, drs,
                                     drs, _ptr(dsink), _stream(stream))
    _check("attn_sink_bwd_strided", rc)
    return (dqkv.reshape(shape4) if shape4 is not None else dqkv), dsink


def attn_sink_bwd_kvpacked(q, kv, sink, out, lse, dout, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                           max_seqlen_k, win_first=0, win_last=0, causal=True, scale=0.0, dq=None, dkv=None,
                           dsink=None, stream=None):
    """Backward of attn_sink_fwd_kvpacked; returns (dq, dkv, dsink or None), dkv in
    the (Tk, 2, hkv, d) layout of kv.  Rows of dkv past every request's last key
    are not written (pass a zeroed ``dkv`` if kv has such rows)."""
    for t, n in ((q, "q"), (kv, "kv"), (out, "out"), (dout, "dout")):
        _need(t, torch.bfloat16, n)
    _need(sink, torch.float32, "sink")
    _need(lse, torch.float32, "lse")
    tq, hq, d = q.shape
    tk, _, hkv, _ = kv.shape
    dq = torch.empty_like(q) if dq is None else dq
    dkv = torch.empty_like(kv) if dkv is None else dkv
    _need(dkv, torch.bfloat16, "dkv")
    if sink is not None and dsink is None:
        dsink = torch.empty_like(sink)
    kp, rs = _row_view(kv.reshape(tk, 2 * hkv, d), 0, hkv, d)
    vp, _ = _row_view(kv.reshape(tk, 2 * hkv, d), hkv, hkv, d)
    dkp, drs = _row_view(dkv.reshape(tk, 2 * hkv, d), 0, hkv, d)
    dvp, _ = _row_view(dkv.reshape(tk, 2 * hkv, d), hkv, hkv, d)
    rc = lib().attn_sink_bwd_strided(_ptr(q), kp, vp, 0, rs, rs, _ptr(sink), _ptr(out), _ptr(lse), _ptr(dout),
                                     _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), cu_seqlens_q.numel() - 1, tq, tk, hq,
                                     hkv, d, int(max_seqlen_q), int(max_seqlen_k), int(win_first),
                                     int(win_last), 1 if causal else 0, float(scale), _ptr(dq), dkp, dvp, 0, drs,
                                     drs, _ptr(dsink), _stream(stream))
    _check("attn_sink_bwd_strided", rc)
    return dq, dkv, dsink


def attn_sink_kv_append(k_new, v_new, k_cache, v_cache, page_table, seqlens, cu_new=None,
                        max_new=None, stream=None):
    """Writes the new K/V rows into the paged caches in place (see the C header)."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n)
    _need(page_table, torch.int32, "page_table")
    _need(seqlens, torch.int32, "seqlens")
    _need(cu_new, torch.int32, "cu_new")
    npages, ps, hkv, d = k_cache.shape
    B = seqlens.numel()
    if max_new is None:
        max_new = 1 if cu_new is None else int((cu_new[1:] - cu_new[:-1]).max()) if B else 0
    rc = lib().attn_sink_kv_append(_ptr(k_new), _ptr(v_new), _ptr(cu_new), _ptr(seqlens), _ptr(page_table),
                                   page_table.shape[1], B, hkv, d, ps, npages, int(max_new), _ptr(k_cache),
                                   _ptr(v_cache), _stream(stream))
    _check("attn_sink_kv_append", rc)
    return k_cache, v_cache


def attn_sink_decode_paged_append(q, k_new, v_new, k_cache, v_cache, page_table, seqlens, sink=None,
                                  win_first=0, win_last=0, scale=0.0, out=None, lse=None,
                                  return_lse=True, stream=None):
    """Paged decode with the new token's K/V (k_new, v_new: (B, Hkv, d)) written into
    the caches first, in the same call."""
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n)
    _need(page_table, torch.int32, "page_table")
    _need(seqlens, torch.int32, "seqlens")
    _need(sink, torch.float32, "sink")
    B, hq, d = q.shape
    npages, ps, hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, hq), dtype=torch.float32, device=q.device)
    rc = lib().attn_sink_decode_paged_append(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                             _ptr(page_table), page_table.shape[1], _ptr(seqlens), B, hq, hkv, d,
                                             ps, npages, _ptr(sink), int(win_first), int(win_last), float(scale),
                                             _ptr(out), _ptr(lse), _stream(stream))
    _check("attn_sink_decode_paged_append", rc)
    return out, lse


def attn_sink_fwd_paged(q, k_cache, v_cache, page_table, cu_seqlens_q, seqlens_k, max_seqlen_q,
                        max_seqlen_k, sink=None, k_new=None, v_new=None, win_first=0, win_last=0,
                        causal=True, scale=0.0, out=None, lse=None, return_lse=True, stream=None):
    """Varlen extend against a paged K/V cache; with k_new/v_new the chunk's K/V
    are appended into the cache first.  Returns (out, lse)."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (k_new, "k_new"), (v_new, "v_new")):
        _need(t, torch.bfloat16, n)
    _need(page_table, torch.int32, "page_table")
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q")
    _need(seqlens_k, torch.int32, "seqlens_k")
    _need(sink, torch.float32, "sink")
    tq, hq, d = q.shape
    npages, ps, hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((hq, tq), dtype=torch.float32, device=q.device)
    rc = lib().attn_sink_fwd_paged(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(page_table), page_table.shape[1], _ptr(cu_seqlens_q), _ptr(seqlens_k),
                                   cu_seqlens_q.numel() - 1, tq, hq, hkv, d, ps, npages, int(max_seqlen_q),
                                   int(max_seqlen_k), _ptr(sink), int(win_first), int(win_last),
                                   1 if causal else 0, float(scale), _ptr(out), _ptr(lse), _stream(stream))
    _check("attn_sink_fwd_paged", rc)
    return out, lse


def attn_sink_bwd(q, k, v, sink, out, lse, dout, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                  max_seqlen_k, win_first=0, win_last=0, causal=True, scale=0.0, dq=None, dk=None,
                  dv=None, dsink=None, stream=None):
    """Backward with the sink's gradient; returns (dq, dk, dv, dsink or None)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _need(t, torch.bfloat16, n)
    _need(sink, torch.float32, "sink")
    _need(lse, torch.float32, "lse")
    tq, hq, d = q.shape
    hkv = k.shape[1]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if sink is not None and dsink is None:
        dsink = torch.empty_like(sink)
    rc = lib().attn_sink_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(sink), _ptr(out), _ptr(lse), _ptr(dout),
                             _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), cu_seqlens_q.numel() - 1, tq,
                             k.shape[0], hq, hkv, d, int(max_seqlen_q), int(max_seqlen_k), int(win_first),
                             int(win_last), 1 if causal else 0, float(scale), _ptr(dq), _ptr(dk),
                             _ptr(dv), _ptr(dsink), _stream(stream))
    _check("attn_sink_bwd", rc)
    return dq, dk, dv, dsink


def attn_sink_visible_ranges(seqlens, win_first, win_last, stream=None):
    _need(seqlens, torch.int32, "seqlens")
    B = seqlens.numel()
    ranges = torch.empty((B, 4), dtype=torch.int32, device=seqlens.device)
    rc = lib().attn_sink_visible_ranges(_ptr(seqlens), B, int(win_first), int(win_last),
                                        _ptr(ranges), _stream(stream))
    _check("attn_sink_visible_ranges", rc)
    return ranges


def attn_sink_visible_slots(seqlens, page_table, page_size, num_pages, win_first, win_last,
                            max_visible, stream=None):
    _need(seqlens, torch.int32, "seqlens")
    _need(page_table, torch.int32, "page_table")
    B = seqlens.numel()
    slots = torch.empty((B, max_visible), dtype=torch.int32, device=seqlens.device)
    rc = lib().attn_sink_visible_slots(_ptr(seqlens), _ptr(page_table), page_table.shape[1], B,
                                       int(page_size), int(num_pages), int(win_first),
                                       int(win_last), _ptr(slots), int(max_visible),
                                       _stream(stream))
    _check("attn_sink_visible_slots", rc)
    return slots


def attn_sink_selftest_wait(complete, stream=None):
    """One single-thread kernel waits on an mbarrier: completed first (returns at
    once) or never completed (gives up after the wait limit and sets DEV_TIMEOUT,
    read by device_status)."""
    _check("attn_sink_selftest_wait", lib().attn_sink_selftest_wait(1 if complete else 0, _stream(stream)))


def device_status(stream=None) -> int:
    rc = lib().attn_sink_device_status(_stream(stream))
    if rc < 0:
        _check("attn_sink_device_status", rc)
    return rc

"""Autograd functions over the C-ABI forward and backward.

The flash-attention PR "feat: Implement Sink Attention" (Key Changes) adds a
learnable per-head sink, shape (nheads,), to the attention functions, the
variable-length ones included, and returns its gradient from the backward.
These functions give the same training-side API on top of ``attn_sink_fwd`` /
``attn_sink_bwd``: each forward calls the library's forward, each backward the
library's backward (which also yields the sink's gradient).  Only arguments
are marshalled here; the computation runs in the library's kernels.

Tensors: q (total_q, Hq, d), k / v (total_k, Hkv, d) bf16 CUDA, contiguous;
``learnable_sink`` (Hq,) fp32 CUDA or None; cu_seqlens int32 CUDA.  LSE is
returned without a gradient (its backward contribution is not defined here).
"""
import torch

from . import _lib


def _scale(softmax_scale):
    return 0.0 if softmax_scale is None else float(softmax_scale)


class _AttnSinkVarlen(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, sink, cu_q, cu_k, max_q, max_k, causal, win_first, win_last, scale):
        out, lse = _lib.attn_sink_fwd(q, k, v, sink, cu_q, cu_k, max_q, max_k, win_first, win_last,
                                      causal, scale)
        ctx.save_for_backward(q, k, v, sink, out, lse, cu_q, cu_k)
        ctx.args = (max_q, max_k, win_first, win_last, causal, scale)
        ctx.mark_non_differentiable(lse)
        return out, lse

    @staticmethod
    def backward(ctx, dout, _dlse):
        q, k, v, sink, out, lse, cu_q, cu_k = ctx.saved_tensors
        max_q, max_k, win_first, win_last, causal, scale = ctx.args
        dq, dk, dv, dsink = _lib.attn_sink_bwd(q, k, v, sink, out, lse, dout.contiguous(), cu_q, cu_k,
                                               max_q, max_k, win_first, win_last, causal, scale)
        if sink is None or not ctx.needs_input_grad[3]:
            dsink = None
        return dq, dk, dv, dsink, None, None, None, None, None, None, None, None


class _AttnSinkVarlenQKVPacked(torch.autograd.Function):
    @staticmethod
    def forward(ctx, qkv, hkv, sink, cu, max_s, causal, win_first, win_last, scale):
        out, lse = _lib.attn_sink_fwd_qkvpacked(qkv, hkv, sink, cu, max_s, win_first, win_last, causal, scale)
        ctx.save_for_backward(qkv, sink, out, lse, cu)
        ctx.args = (hkv, max_s, win_first, win_last, causal, scale)
        ctx.mark_non_differentiable(lse)
        return out, lse

    @staticmethod
    def backward(ctx, dout, _dlse):
        qkv, sink, out, lse, cu = ctx.saved_tensors
        hkv, max_s, win_first, win_last, causal, scale = ctx.args
        # zeroed: rows past the last sequence's end (padding) are not written
        dqkv, dsink = _lib.attn_sink_bwd_qkvpacked(qkv, hkv, sink, out, lse, dout.contiguous(), cu, max_s,
                                                   win_first, win_last, causal, scale,
                                                   dqkv=torch.zeros_like(qkv))
        if sink is None or not ctx.needs_input_grad[2]:
            dsink = None
        return dqkv, None, dsink, None, None, None, None, None, None


class _AttnSinkVarlenKVPacked(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, kv, sink, cu_q, cu_k, max_q, max_k, causal, win_first, win_last, scale):
        out, lse = _lib.attn_sink_fwd_kvpacked(q, kv, sink, cu_q, cu_k, max_q, max_k, win_first, win_last,
                                               causal, scale)
        ctx.save_for_backward(q, kv, sink, out, lse, cu_q, cu_k)
        ctx.args = (max_q, max_k, win_first, win_last, causal, scale)
        ctx.mark_non_differentiable(lse)
        return out, lse

    @staticmethod
    def backward(ctx, dout, _dlse):
        q, kv, sink, out, lse, cu_q, cu_k = ctx.saved_tensors
        max_q, max_k, win_first, win_last, causal, scale = ctx.args
        # zeroed: rows past the last sequence's end (padding) are not written
        dq, dkv, dsink = _lib.attn_sink_bwd_kvpacked(q, kv, sink, out, lse, dout.contiguous(), cu_q, cu_k, max_q,
                                                     max_k, win_first, win_last, causal, scale,
                                                     dkv=torch.zeros_like(kv))
        if sink is None or not ctx.needs_input_grad[2]:
            dsink = None
        return dq, dkv, dsink, None, None, None, None, None, None, None, None


def attn_sink_varlen_func(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                          learnable_sink=None, causal=True, win_first=0, win_last=0, softmax_scale=None,
                          return_lse=False):
    """Variable-length attention with a learnable sink; differentiable in q, k,
    v and ``learnable_sink``.  Returns out (total_q, Hq, d), and LSE (Hq,
    total_q) fp32 as well when ``return_lse``."""
    out, lse = _AttnSinkVarlen.apply(q, k, v, learnable_sink, cu_seqlens_q, cu_seqlens_k, int(max_seqlen_q),
                                     int(max_seqlen_k), bool(causal), int(win_first), int(win_last),
                                     _scale(softmax_scale))
    return (out, lse) if return_lse else out


def attn_sink_func(q, k, v, learnable_sink=None, causal=True, win_first=0, win_last=0, softmax_scale=None,
                   return_lse=False):
    """Equal-length batches: q (B, Sq, Hq, d), k / v (B, Sk, Hkv, d).  The
    batch is passed to the library as B sequences of Sq queries and Sk keys
    (bottom-right causal alignment when Sq < Sk).  Returns out (B, Sq, Hq, d),
    and LSE (Hq, B * Sq) when ``return_lse``."""
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise TypeError("attn_sink_func takes (batch, seqlen, heads, head_dim) tensors")
    B, sq, hq, d = q.shape
    sk = k.shape[1]
    cu_q, cu_k = _cu(B, sq, q.device), _cu(B, sk, q.device)
    out, lse = _AttnSinkVarlen.apply(q.reshape(B * sq, hq, d), k.reshape(B * sk, k.shape[2], d),
                                     v.reshape(B * sk, v.shape[2], d), learnable_sink, cu_q, cu_k, sq, sk,
                                     bool(causal), int(win_first), int(win_last), _scale(softmax_scale))
    out = out.reshape(B, sq, hq, d)
    return (out, lse) if return_lse else out


def attn_sink_varlen_qkvpacked_func(qkv, cu_seqlens, max_seqlen, hkv=None, learnable_sink=None, causal=True,
                                    win_first=0, win_last=0, softmax_scale=None, return_lse=False):
    """Self-attention on a packed buffer: qkv (total, 3, H, d) (then hkv = H), or
    (total, Hq + 2 Hkv, d) with ``hkv`` given; differentiable in qkv and
    ``learnable_sink``.  The gradient comes back in the layout of qkv."""
    if qkv.dim() == 4:
        if qkv.shape[1] != 3:
            raise TypeError("a 4-D qkv must be (total, 3, heads, head_dim)")
        hkv = qkv.shape[2]
    elif hkv is None:
        raise TypeError("hkv is required for a (total, Hq + 2 Hkv, head_dim) qkv")
    out, lse = _AttnSinkVarlenQKVPacked.apply(qkv, int(hkv), learnable_sink, cu_seqlens, int(max_seqlen),
                                              bool(causal), int(win_first), int(win_last), _scale(softmax_scale))
    return (out, lse) if return_lse else out


def attn_sink_varlen_kvpacked_func(q, kv, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                                   learnable_sink=None, causal=True, win_first=0, win_last=0, softmax_scale=None,
                                   return_lse=False):
    """q (total_q, Hq, d) against a packed kv (total_k, 2, Hkv, d); differentiable in
    q, kv and ``learnable_sink``.  The gradient of kv comes back in its layout."""
    if kv.dim() != 4 or kv.shape[1] != 2:
        raise TypeError("kv must be (total_k, 2, heads, head_dim)")
    out, lse = _AttnSinkVarlenKVPacked.apply(q, kv, learnable_sink, cu_seqlens_q, cu_seqlens_k, int(max_seqlen_q),
                                             int(max_seqlen_k), bool(causal), int(win_first), int(win_last),
                                             _scale(softmax_scale))
    return (out, lse) if return_lse else out


def _cu(batch, seqlen, device):
    return torch.arange(0, (batch + 1) * seqlen, seqlen, dtype=torch.int32, device=device)


def attn_sink_qkvpacked_func(qkv, learnable_sink=None, causal=True, win_first=0, win_last=0, softmax_scale=None,
                             return_lse=False):
    """Equal-length batches of packed self-attention: qkv (B, S, 3, H, d).
    Returns out (B, S, H, d) (and LSE (H, B * S) when ``return_lse``)."""
    if qkv.dim() != 5 or qkv.shape[2] != 3:
        raise TypeError("qkv must be (batch, seqlen, 3, heads, head_dim)")
    B, S, _, H, d = qkv.shape
    out, lse = attn_sink_varlen_qkvpacked_func(qkv.reshape(B * S, 3, H, d), _cu(B, S, qkv.device), S,
                                               learnable_sink=learnable_sink, causal=causal, win_first=win_first,
                                               win_last=win_last, softmax_scale=softmax_scale, return_lse=True)
    out = out.reshape(B, S, H, d)
    return (out, lse) if return_lse else out


def attn_sink_kvpacked_func(q, kv, learnable_sink=None, causal=True, win_first=0, win_last=0, softmax_scale=None,
                            return_lse=False):
    """Equal-length batches: q (B, Sq, Hq, d) against kv (B, Sk, 2, Hkv, d).
    Returns out (B, Sq, Hq, d) (and LSE (Hq, B * Sq) when ``return_lse``)."""
    if q.dim() != 4 or kv.dim() != 5 or kv.shape[2] != 2:
        raise TypeError("q must be (batch, seqlen, heads, head_dim) and kv (batch, seqlen, 2, heads, head_dim)")
    B, sq, hq, d = q.shape
    sk, hkv = kv.shape[1], kv.shape[3]
    out, lse = attn_sink_varlen_kvpacked_func(q.reshape(B * sq, hq, d), kv.reshape(B * sk, 2, hkv, d),
                                              _cu(B, sq, q.device), _cu(B, sk, q.device), sq, sk,
                                              learnable_sink=learnable_sink, causal=causal, win_first=win_first,
                                              win_last=win_last, softmax_scale=softmax_scale, return_lse=True)
    out = out.reshape(B, sq, hq, d)
    return (out, lse) if return_lse else out

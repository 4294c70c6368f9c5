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
        dqkv, dsink = _lib.attn_sink_bwd_qkvpacked(qkv, hkv, sink, out, lse, dout.contiguous(), cu, max_s,
                                                   win_first, win_last, causal, scale)
        if sink is None or not ctx.needs_input_grad[2]:
            dsink = None
        return dqkv, None, dsink, None, None, None, None, None, None


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
    dev = q.device
    cu_q = torch.arange(0, (B + 1) * sq, sq, dtype=torch.int32, device=dev)
    cu_k = torch.arange(0, (B + 1) * sk, sk, dtype=torch.int32, device=dev)
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

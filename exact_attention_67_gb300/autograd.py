"""Differentiable attention for PyTorch training code.

``attention`` takes [B, H, N, d] tensors; ``flash_attn_func`` takes the
[batch, seqlen, heads, head_dim] layout of the flash_attn_func example in
"提示词再优也救不了的性能黑洞…" (第一章) and returns the output in that layout.
Both run the library's forward and, on ``.backward()``, its backward (the
gradients of softmax(scale Q K^T [+ causal mask]) V); nothing here computes.
"""
from __future__ import annotations

import torch

from . import backward as _backward
from . import forward as _forward


class _Attention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, causal: bool, scale, window: int, fp32_o: bool):
        if fp32_o:
            o, lse, o32 = _forward(q, k, v, causal, scale, window=window, fp32_o=True)
            ctx.save_for_backward(q, k, v, o32, lse)
        else:
            o, lse = _forward(q, k, v, causal, scale, window=window)
            ctx.save_for_backward(q, k, v, o, lse)
        ctx.causal, ctx.scale, ctx.window, ctx.fp32_o = causal, scale, window, fp32_o
        return o

    @staticmethod
    @torch.autograd.function.once_differentiable
    def backward(ctx, do):
        q, k, v, o_saved, lse = ctx.saved_tensors
        # The library reads dO through its strides (d contiguous, other strides
        # multiples of 8 elements, nonzero) from a 16-byte-aligned address: an
        # expanded, oddly strided or offset gradient (e.g. from
        # out.sum().backward(), or a slice of a larger buffer) is made
        # contiguous first.
        if (do.stride(-1) != 1 or any(s == 0 or s % 8 for s in do.stride()[:-1]) or
                do.data_ptr() % 16 != 0):
            do = do.contiguous()
        if ctx.fp32_o:
            dq, dk, dv = _backward(q, k, v, None, lse, do, ctx.causal, ctx.scale, window=ctx.window, o32=o_saved)
        else:
            dq, dk, dv = _backward(q, k, v, o_saved, lse, do, ctx.causal, ctx.scale, window=ctx.window)
        return dq, dk, dv, None, None, None, None


def attention(q, k, v, causal: bool = False, scale: float | None = None, window: int = 0, fp32_o: bool = False):
    """O = softmax(scale Q K^T [+ causal mask, sliding window]) V for [B, H, N, d]
    bf16/f16 CUDA tensors (any layout with d contiguous), differentiable in q,
    k and v.  scale defaults to 1/sqrt(d).  ``fp32_o`` keeps an fp32 copy of O
    for the backward's row terms (B*H*N*d*4 bytes until backward): accurate
    gradients also on rows whose softmax is nearly one-hot."""
    return _Attention.apply(q, k, v, bool(causal), scale, int(window), bool(fp32_o))


def flash_attn_func(q, k, v, dropout_p: float = 0.0, softmax_scale: float | None = None, causal: bool = False):
    """q, k, v: [batch, seqlen, heads, head_dim]; returns O in that layout.
    Differentiable.  Only dropout_p = 0 is supported (the method is exact
    attention; there is no dropout)."""
    if dropout_p != 0.0:
        raise ValueError("dropout is not supported (dropout_p must be 0)")
    o = attention(q.transpose(1, 2), k.transpose(1, 2), v.transpose(1, 2), causal, softmax_scale)
    return o.transpose(1, 2)

"""exact_attention_67_gb300 -- fused exact attention for NVIDIA GB300 (sm_103a).

O = softmax(scale * Q K^T [+ causal mask]) V in one fused TMA + tcgen05 kernel
with an online softmax (S and P never leave the chip), and its gradient with
tile-by-tile recomputation from the stored logsumexp.  The C ABI is in
``include/exattn.h``; ``attn_fwd`` / ``attn_bwd`` here are its ctypes binding
(same names, argument marshalling only) and :func:`forward` /
:func:`backward` allocate the outputs with PyTorch.

The helpers (forward, backward, their varlen and decode forms, attention)
also watch the kernels' watchdog without synchronising: each call queues a
copy of the device's watchdog word into page-locked memory after its
launches, and the next call raises ExattnError (EXATTN_ERR_TIMEOUT) if a
completed copy shows that a bounded wait gave up.
"""
from __future__ import annotations

import math

from ._lib import (EXPORTS, ExattnError, Strides, attn_bwd, attn_bwd_d_and_dq, attn_bwd_dkdv, attn_bwd_dq, attn_bwd_ex,
                   attn_bwd_o32, attn_fwd_o32, attn_bwd_preprocess, attn_bwd_varlen, attn_bwd_workspace_size, attn_fwd, attn_fwd_decode, attn_fwd_bwd_host,
                   attn_fwd_bwd_host_workspace_size, attn_fwd_decode_workspace_size, attn_fwd_ex, attn_fwd_varlen,
                   device_error, library_path, load, status_string, version, watchdog_check, watchdog_poll)
from .host import HostStep, fwd_bwd_from_host

__all__ = ["attn_fwd", "attn_bwd", "attn_bwd_workspace_size", "attn_bwd_preprocess", "attn_bwd_dkdv",
           "attn_bwd_dq", "attn_bwd_d_and_dq", "attn_fwd_ex", "attn_bwd_ex", "attn_fwd_o32", "attn_bwd_o32",
           "attn_fwd_varlen", "attn_bwd_varlen", "Strides", "forward", "backward", "forward_varlen", "backward_varlen", "attn_fwd_decode", "attn_fwd_decode_workspace_size",
           "forward_decode", "fwd_bwd_from_host", "HostStep", "attn_fwd_bwd_host",
           "attn_fwd_bwd_host_workspace_size", "attention", "flash_attn_func", "device_error",
           "watchdog_check", "watchdog_poll", "status_string", "version", "load", "library_path", "ExattnError",
           "EXPORTS"]


def _default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def _plain(*ts) -> bool:
    import torch
    return all(t.dtype == torch.bfloat16 and t.is_contiguous() for t in ts)


def forward(q, k, v, causal: bool = False, scale: float | None = None, stream=None, window: int = 0,
            fp32_o: bool = False):
    """Allocate O (same type and memory layout as q) and lse (fp32) with torch
    and run ``attn_fwd`` (contiguous bf16) or ``attn_fwd_ex`` (f16 or strided
    [B, H, N, d] views, e.g. ``x.transpose(1, 2)`` of a [B, N, H, d] tensor, or
    a sliding ``window`` > 0).  With ``fp32_o`` it runs ``attn_fwd_o32`` and
    returns (O, lse, O in fp32) for ``backward(..., o32=...)``."""
    import torch
    B, H, N, d = q.shape
    s = _default_scale(d) if scale is None else scale
    watchdog_check(q.device)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if fp32_o:
        o32 = torch.empty((B, H, N, d), dtype=torch.float32, device=q.device)
        attn_fwd_o32(q, k, v, o, lse, o32, causal, s, stream, window)
        watchdog_poll(q.device, stream)
        return o, lse, o32
    if window == 0 and _plain(q, k, v, o):
        attn_fwd(q, k, v, o, lse, causal, s, stream)
    else:
        attn_fwd_ex(q, k, v, o, lse, causal, s, stream, window)
    watchdog_poll(q.device, stream)
    return o, lse


def backward(q, k, v, o, lse, dO, causal: bool = False, scale: float | None = None, stream=None,
             workspace=None, window: int = 0, o32=None):
    """Allocate dQ, dK, dV (like q, k, v) and the workspace unless given, and run
    ``attn_bwd`` (contiguous bf16) or ``attn_bwd_ex``; with ``o32`` (from
    ``forward(..., fp32_o=True)``) ``attn_bwd_o32``, which takes the row terms
    D_i from it and does not read ``o``."""
    import torch
    B, H, N, d = q.shape
    s = _default_scale(d) if scale is None else scale
    watchdog_check(q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if workspace is None:
        nbytes = attn_bwd_workspace_size(B, H, N, d, causal)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    if o32 is not None:
        attn_bwd_o32(q, k, v, o32, dO, lse, dq, dk, dv, causal, s, workspace, stream, window)
    elif window == 0 and _plain(q, k, v, o, dO, dq, dk, dv):
        attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, causal, s, workspace, stream)
    else:
        attn_bwd_ex(q, k, v, o, dO, lse, dq, dk, dv, causal, s, workspace, stream, window)
    watchdog_poll(q.device, stream)
    return dq, dk, dv


def forward_varlen(q, k, v, cu_seqlens, max_seqlen: int, causal: bool = False, scale: float | None = None,
                   stream=None, window: int = 0):
    """Packed variable-length forward: q, k, v [total, H, d]; returns O (like q)
    and lse fp32 [H, total]."""
    import torch
    total, H, d = q.shape
    s = _default_scale(d) if scale is None else scale
    watchdog_check(q.device)
    o = torch.empty_like(q)
    lse = torch.empty((H, total), dtype=torch.float32, device=q.device)
    attn_fwd_varlen(q, k, v, o, lse, cu_seqlens, max_seqlen, causal, s, stream, window)
    watchdog_poll(q.device, stream)
    return o, lse


def backward_varlen(q, k, v, o, lse, dO, cu_seqlens, max_seqlen: int, causal: bool = False,
                    scale: float | None = None, stream=None, window: int = 0, workspace=None):
    """Packed variable-length backward: returns dQ, dK, dV (like q, k, v)."""
    import torch
    total, H, d = q.shape
    s = _default_scale(d) if scale is None else scale
    watchdog_check(q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if workspace is None:
        workspace = torch.empty(attn_bwd_workspace_size(1, H, total, d, causal), dtype=torch.uint8, device=q.device)
    attn_bwd_varlen(q, k, v, o, dO, lse, dq, dk, dv, cu_seqlens, max_seqlen, causal, s, workspace, stream, window)
    watchdog_poll(q.device, stream)
    return dq, dk, dv


def forward_decode(q, k, v, causal: bool = False, scale: float | None = None, stream=None, window: int = 0):
    """Decode-shaped forward: q [B, H, Nq, d] against k, v [B, H, Nk, d], the
    queries aligned to the last Nq keys; returns O (like q) and lse [B, H, Nq]."""
    import torch
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    s = _default_scale(d) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    watchdog_check(q.device)
    nbytes = attn_fwd_decode_workspace_size(B, H, Nq, Nk, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device) if nbytes else None
    attn_fwd_decode(q, k, v, o, lse, causal, s, ws, stream, window)
    watchdog_poll(q.device, stream)
    return o, lse


from .autograd import attention, flash_attn_func  # noqa: E402  (uses forward/backward above)

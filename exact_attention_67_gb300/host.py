"""Attention forward + backward on host-resident tensors, with the host <-> device
copies overlapped with the kernels.

The (batch, head) problems are independent, so they are processed in groups:
while group i runs on the device, the inputs of later groups are copied in on
one stream and the results of group i-1 are copied out on another.  The copies
and the stream plumbing are PyTorch's; every attention step runs in the
library's kernels (the forward, then the backward stage by stage so that O and
lse, then dK and dV, leave while later stages run).
"""
from __future__ import annotations

import math

import torch

from ._lib import (attn_bwd_dkdv, attn_bwd_dq, attn_bwd_ex, attn_bwd_preprocess, attn_bwd_workspace_size, attn_fwd,
                   attn_fwd_ex)

_streams: dict = {}


def _side_streams(device, n: int):
    """n streams of `device`, created once and reused."""
    key = torch.device(device).index
    have = _streams.setdefault(key, [])
    while len(have) < n:
        have.append(torch.cuda.Stream(device=device))
    return have[:n]


def fwd_bwd_from_host(q, k, v, dO, causal: bool = False, scale: float | None = None, groups: int = 2,
                      device="cuda:0", out=None, streams: int = 1):
    """q, k, v, dO: host tensors [B, H, N, d] (bf16 or f16, contiguous; pinned
    for the copies to overlap).  Returns host (O, lse, dQ, dK, dV), written into
    ``out`` (five pinned host tensors of those shapes) when given.  Asynchronous
    with respect to the host: synchronise the device's current stream before
    reading the results.  ``groups`` (at most B*H) sets how many groups of
    (batch, head) problems the copies are overlapped with; with ``streams`` >
    1 consecutive groups run on that many compute streams, so that the
    kernels of small groups share the GPU (each CTA holds a whole SM, so
    concurrent kernels split the SMs between them)."""
    if q.dim() != 4:
        raise ValueError("q must be [B, H, N, d]")
    B, H, N, d = q.shape
    BH = B * H
    for name, t in (("q", q), ("k", k), ("v", v), ("dO", dO)):
        if t.shape != q.shape or t.dtype != q.dtype or t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError(f"{name}: expected a contiguous host tensor like q ({tuple(q.shape)}, {q.dtype})")
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("q, k, v, dO must be bf16 or f16")
    s = 1.0 / math.sqrt(d) if scale is None else scale
    groups = max(1, min(int(groups), BH))
    want = ((q.shape, q.dtype), ((B, H, N), torch.float32), (q.shape, q.dtype), (q.shape, q.dtype), (q.shape, q.dtype))
    if out is not None and (len(out) != 5 or any(
            t.shape != sh or t.dtype != dt or t.device.type != "cpu" or not t.is_contiguous()
            for t, (sh, dt) in zip(out, want))):
        raise ValueError("out: expected contiguous host tensors O, lse (fp32 [B, H, N]), dQ, dK, dV")
    dev = torch.device(device)
    comp = torch.cuda.current_stream(dev)
    n_cs = max(1, min(int(streams), groups))
    side = _side_streams(dev, 2 + n_cs - 1)
    s_in, s_out = side[0], side[1]
    cs = [comp] + side[2:]  # compute stream of group i: cs[i % n_cs]
    flat_in = [t.view(BH, N, d) for t in (q, k, v, dO)]
    if out is None:
        out = tuple(torch.empty(sh, dtype=dt).pin_memory() for sh, dt in want)
    flat_out = [t.view(BH, *t.shape[2:]) for t in out]
    d_in = [torch.empty((BH, N, d), dtype=q.dtype, device=dev) for _ in range(4)]
    d_out = [torch.empty((BH, N, d), dtype=q.dtype, device=dev), torch.empty((BH, N), dtype=torch.float32, device=dev)]
    d_out += [torch.empty((BH, N, d), dtype=q.dtype, device=dev) for _ in range(3)]
    bounds = [(i * BH) // groups for i in range(groups + 1)]
    largest = max(bounds[i + 1] - bounds[i] for i in range(groups))
    ws_bytes = attn_bwd_workspace_size(1, largest, N, d, causal)
    ws_bytes = (ws_bytes + 255) // 256 * 256
    ws_all = torch.empty(ws_bytes * n_cs, dtype=torch.uint8, device=dev)  # one workspace per compute stream
    for t in d_in:
        t.record_stream(s_in)
    for t in d_out:
        t.record_stream(s_out)
    for c in cs[1:]:
        for t in d_in + d_out + [ws_all]:
            t.record_stream(c)
        c.wait_stream(comp)
    s_in.wait_stream(comp)  # earlier work on the current stream may still use recycled memory
    # Inputs in use order: Q, K, V of a group (the forward), then its dO (the backward).
    ev_qkv, ev_do = [], []
    with torch.cuda.stream(s_in):
        for i in range(groups):
            a, b = bounds[i], bounds[i + 1]
            for src, dst in zip(flat_in[:3], d_in[:3]):
                dst[a:b].copy_(src[a:b], non_blocking=True)
            e = torch.cuda.Event()
            e.record(s_in)
            ev_qkv.append(e)
            d_in[3][a:b].copy_(flat_in[3][a:b], non_blocking=True)
            e = torch.cuda.Event()
            e.record(s_in)
            ev_do.append(e)

    def copy_out(idx, a, b, c):
        """After the work queued so far on compute stream c, copy outputs idx of rows [a, b) to the host."""
        e = torch.cuda.Event()
        e.record(c)
        s_out.wait_event(e)
        with torch.cuda.stream(s_out):
            for j in idx:
                flat_out[j][a:b].copy_(d_out[j][a:b], non_blocking=True)

    staged = q.dtype == torch.bfloat16  # the stage calls take bf16; f16 runs the backward as one call
    for i in range(groups):
        a, b = bounds[i], bounds[i + 1]
        c = cs[i % n_cs]
        ws = ws_all[(i % n_cs) * ws_bytes:(i % n_cs + 1) * ws_bytes]
        q_g, k_g, v_g, do_g = (t[a:b].unsqueeze(0) for t in d_in)  # the group as one batch of b - a heads
        o_g, lse_g, dq_g, dk_g, dv_g = (t[a:b].unsqueeze(0) for t in d_out)
        c.wait_event(ev_qkv[i])
        (attn_fwd if staged else attn_fwd_ex)(q_g, k_g, v_g, o_g, lse_g, causal, s, stream=c)
        copy_out((0, 1), a, b, c)  # O and lse leave while the backward runs
        c.wait_event(ev_do[i])
        if staged:
            D = ws[: (b - a) * N * 4].view(torch.float32).view(1, b - a, N)
            attn_bwd_preprocess(o_g, do_g, D, stream=c)
            attn_bwd_dkdv(q_g, k_g, v_g, do_g, lse_g, D, dk_g, dv_g, causal, s, stream=c)
            copy_out((3, 4), a, b, c)  # dK, dV leave while dQ is computed
            attn_bwd_dq(q_g, k_g, v_g, do_g, lse_g, D, dq_g, causal, s, stream=c)
            copy_out((2,), a, b, c)
        else:
            attn_bwd_ex(q_g, k_g, v_g, o_g, do_g, lse_g, dq_g, dk_g, dv_g, causal, s, ws, stream=c)
            copy_out((2, 3, 4), a, b, c)
    for c in cs[1:]:
        comp.wait_stream(c)
    comp.wait_stream(s_out)
    return out


class HostStep:
    """fwd_bwd_from_host captured once as a CUDA graph.

    Each call replays the whole step -- the host -> device copies of q, k, v,
    dO (whatever the pinned host tensors hold at that moment), the kernels and
    the device -> host copies into ``out`` -- with one graph launch instead of
    the host-side work of issuing a few dozen copies, kernels and events.
    The host tensors must stay alive and keep their storage while the step is
    in use.  Results are those of fwd_bwd_from_host (bit for bit)."""

    def __init__(self, q, k, v, dO, causal: bool = False, scale: float | None = None, groups: int = 4,
                 streams: int = 2, device="cuda:0", out=None):
        dev = torch.device(device)
        for t in (q, k, v, dO):
            if not t.is_pinned():
                raise ValueError("HostStep needs pinned host tensors (tensor.pin_memory())")
        args = dict(causal=causal, scale=scale, groups=groups, device=dev, streams=streams)
        if out is None:
            B, H, N, _ = q.shape
            out = (torch.empty_like(q).pin_memory(), torch.empty((B, H, N), dtype=torch.float32).pin_memory(),
                   torch.empty_like(q).pin_memory(), torch.empty_like(k).pin_memory(),
                   torch.empty_like(v).pin_memory())
        self.inputs, self.out = (q, k, v, dO), out
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):  # first calls outside the capture: one-time kernel and stream setup
            for _ in range(2):
                fwd_bwd_from_host(q, k, v, dO, out=out, **args)
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize(dev)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            fwd_bwd_from_host(q, k, v, dO, out=out, **args)
        torch.cuda.synchronize(dev)

    def __call__(self):
        """Run the step on the current stream; returns the host (O, lse, dQ, dK, dV).
        Synchronise before reading them."""
        self.graph.replay()
        return self.out

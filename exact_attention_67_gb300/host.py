"""Attention forward + backward on host-resident tensors, with the host <-> device
copies overlapped with the kernels.

``fwd_bwd_from_host`` is the Python face of the C ABI's ``attn_fwd_bwd_host``:
the library splits the (batch, head) problems into groups and, while one
group's kernels run, copies later groups' inputs in on one stream and earlier
results out on another (O and lse during the backward, dK and dV during dQ).
PyTorch supplies the device workspace and the streams; every copy and kernel
is issued by the library.  ``HostStep`` captures one such call as a CUDA
graph and replays it.
"""
from __future__ import annotations

import math

import torch

from ._lib import attn_fwd_bwd_host, attn_fwd_bwd_host_workspace_size

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
    (batch, head) problems the copies are overlapped with; ``streams`` = 2 runs
    every other group on a second compute stream, so that the kernels of small
    groups share the GPU (each CTA holds a whole SM, so concurrent kernels
    split the SMs between them)."""
    if q.dim() != 4:
        raise ValueError("q must be [B, H, N, d]")
    B, H, N, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v), ("dO", dO)):
        if t.shape != q.shape or t.dtype != q.dtype or t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError(f"{name}: expected a contiguous host tensor like q ({tuple(q.shape)}, {q.dtype})")
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("q, k, v, dO must be bf16 or f16")
    if int(groups) < 1:
        raise ValueError("groups must be >= 1")
    s = 1.0 / math.sqrt(d) if scale is None else scale
    want = ((q.shape, q.dtype), ((B, H, N), torch.float32), (q.shape, q.dtype), (q.shape, q.dtype), (q.shape, q.dtype))
    if out is not None and (len(out) != 5 or any(
            t.shape != sh or t.dtype != dt or t.device.type != "cpu" or not t.is_contiguous()
            for t, (sh, dt) in zip(out, want))):
        raise ValueError("out: expected contiguous host tensors O, lse (fp32 [B, H, N]), dQ, dK, dV")
    dev = torch.device(device)
    if out is None:
        out = tuple(torch.empty(sh, dtype=dt).pin_memory() for sh, dt in want)
    with torch.cuda.device(dev):
        comp = torch.cuda.current_stream(dev)
        two = int(streams) > 1 and int(groups) > 1
        side = _side_streams(dev, 3 if two else 2)
        ws = torch.empty(attn_fwd_bwd_host_workspace_size(B, H, N, d, causal), dtype=torch.uint8, device=dev)
        for st in side:
            ws.record_stream(st)  # the library's copies and kernels on the side streams use it too
        o, lse, dq, dk, dv = out
        attn_fwd_bwd_host(q, k, v, dO, o, lse, dq, dk, dv, causal, s, ws, groups=int(groups), stream=comp,
                          copy_in_stream=side[0], copy_out_stream=side[1], stream2=side[2] if two else None)
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

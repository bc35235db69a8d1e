"""Throughput of the library's wider entry points on one GPU:

    python -m exact_attention_67_gb300.bench_rows [--iters 20]

One JSON line per case: f16 inputs, the [B, N, H, d] layout, a sliding
window, a packed variable-length batch and decode-shaped forwards.  Inputs are
seeded synthetic bf16/f16 N(0, 1), resident on the device; each figure is the
mean device time of ``iters`` back-to-back calls between two CUDA events after
three warm-up calls (the square cases move far more than L2 per call and are
compute-bound); the decode cases run the C ABI call on preallocated buffers,
``iters`` calls captured once as a CUDA graph and replayed, so that the
host's per-call work does not show in calls of a few microseconds.  FLOPs count
only visible (query, key) pairs: 4 d per pair forward, 2.5x that backward.
"""
from __future__ import annotations

import argparse
import json
import os

import torch

from . import attn_fwd_decode, attn_fwd_decode_workspace_size, backward, backward_varlen, forward, forward_varlen
from .synth import seeded_bf16

DEV = torch.device("cuda:0")


def _peaks():
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, 6800.0, "fallback"


def _time_ms(fn, iters: int) -> float:
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(iters):
        fn()
    b.record()
    b.synchronize()
    return a.elapsed_time(b) / iters


def _pairs(nq: int, nk: int, causal: bool, window: int) -> int:
    """Visible (query, key) pairs of one head, queries at the last nq of nk positions."""
    total = 0
    off = nk - nq
    for i in range(nq):
        p = i + off
        lo = max(0, p - window + 1) if window > 0 else 0
        hi = p if causal else (min(nk - 1, p + window - 1) if window > 0 else nk - 1)
        total += max(0, hi - lo + 1)
    return total


def _square(name, B, H, N, d, causal, dtype, layout="bhnd", window=0, iters=20, peak=1.0):
    x = [seeded_bf16((B, H, N, d), 11 + t, 1.0, dtype) for t in range(4)]
    if layout == "bnhd":
        q, k, v, do = (t.transpose(1, 2).contiguous().to(DEV).transpose(1, 2) for t in x)
    else:
        q, k, v, do = (t.to(DEV) for t in x)
    scale = d ** -0.5
    o, lse = forward(q, k, v, causal, scale, window=window)
    t_f = _time_ms(lambda: forward(q, k, v, causal, scale, window=window), iters)
    t_b = _time_ms(lambda: backward(q, k, v, o, lse, do, causal, scale, window=window), iters)
    f = 4.0 * d * _pairs(N, N, causal, window) * B * H
    return {"case": name, "B": B, "H": H, "N": N, "d": d, "causal": causal, "window": window,
            "dtype": str(dtype).replace("torch.", ""), "layout": layout, "fwd_ms": t_f, "bwd_ms": t_b,
            "fwd_tflops": f / t_f / 1e9, "bwd_tflops": 2.5 * f / t_b / 1e9,
            "fwd_bwd_tflops": 3.5 * f / (t_f + t_b) / 1e9, "fwd_pct_peak": f / t_f / 1e9 / peak * 100}


def _varlen(name, lens, H, d, causal, dtype, iters, peak):
    total = sum(lens)
    q, k, v, do = (seeded_bf16((total, H, d), 21 + t, 1.0, dtype).to(DEV) for t in range(4))
    cu = torch.tensor([0] + list(torch.tensor(lens).cumsum(0)), dtype=torch.int32, device=DEV)
    scale = d ** -0.5
    mx = max(lens)
    o, lse = forward_varlen(q, k, v, cu, mx, causal, scale)
    t_f = _time_ms(lambda: forward_varlen(q, k, v, cu, mx, causal, scale), iters)
    t_b = _time_ms(lambda: backward_varlen(q, k, v, o, lse, do, cu, mx, causal, scale), iters)
    f = 4.0 * d * H * sum(_pairs(n, n, causal, 0) for n in lens)
    return {"case": name, "lens": lens, "H": H, "d": d, "causal": causal, "dtype": str(dtype).replace("torch.", ""),
            "fwd_ms": t_f, "bwd_ms": t_b, "fwd_tflops": f / t_f / 1e9, "bwd_tflops": 2.5 * f / t_b / 1e9,
            "fwd_bwd_tflops": 3.5 * f / (t_f + t_b) / 1e9, "fwd_pct_peak": f / t_f / 1e9 / peak * 100}


def _time_graph_ms(fn, iters: int) -> float:
    """Mean device time of ``iters`` calls captured once as a CUDA graph and
    replayed: back-to-back launches with no host work between them, for
    calls too short to hide the host's per-call overhead."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(iters):
            fn()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    g.replay()
    b.record()
    b.synchronize()
    return a.elapsed_time(b) / iters


def _decode(name, B, H, Nq, Nk, d, iters, hbm):
    q = seeded_bf16((B, H, Nq, d), 31, 1.0).to(DEV)
    k = seeded_bf16((B, H, Nk, d), 32, 1.0).to(DEV)
    v = seeded_bf16((B, H, Nk, d), 33, 1.0).to(DEV)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=DEV)
    nws = attn_fwd_decode_workspace_size(B, H, Nq, Nk, d)
    ws = torch.empty(nws, dtype=torch.uint8, device=DEV) if nws else None
    # The C ABI call on preallocated buffers (what forward_decode runs, minus
    # its allocations and watchdog poll), replayed from a CUDA graph.
    t = _time_graph_ms(lambda: attn_fwd_decode(q, k, v, o, lse, True, d ** -0.5, ws), iters)
    nbytes = 2.0 * B * H * Nk * d * 2 + 2.0 * B * H * Nq * d * 2  # K, V read; Q read, O written
    return {"case": name, "B": B, "H": H, "Nq": Nq, "Nk": Nk, "d": d, "causal": True, "ms": t,
            "gbs": nbytes / t / 1e6, "pct_hbm": nbytes / t / 1e6 / hbm * 100,
            "workspace_bytes": attn_fwd_decode_workspace_size(B, H, Nq, Nk, d)}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--iters", type=int, default=20)
    a = ap.parse_args(argv)
    peak, hbm, src = _peaks()
    rows = [
        _square("bf16 [B,H,N,d] (reference point)", 1, 16, 8192, 128, True, torch.bfloat16, iters=a.iters, peak=peak),
        _square("f16 [B,H,N,d]", 1, 16, 8192, 128, True, torch.float16, iters=a.iters, peak=peak),
        _square("bf16 [B,N,H,d]", 1, 16, 8192, 128, True, torch.bfloat16, layout="bnhd", iters=a.iters, peak=peak),
        _square("bf16 sliding window 1024", 1, 16, 8192, 128, True, torch.bfloat16, window=1024, iters=a.iters,
                peak=peak),
        _varlen("bf16 packed varlen", [8192, 4096, 4096, 2048, 1024, 512, 256, 128] * 2, 16, 128, True,
                torch.bfloat16, a.iters, peak),
        _decode("decode Nq=1", 4, 32, 1, 32768, 128, a.iters, hbm),
        _decode("decode Nq=1, one head", 1, 1, 1, 131072, 128, a.iters, hbm),
        _decode("decode Nq=16", 8, 16, 16, 16384, 128, a.iters, hbm),
    ]
    for r in rows:
        r["peak_source"] = src
        print(json.dumps(r))


if __name__ == "__main__":
    main()

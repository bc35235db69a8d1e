"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers; it holds none of the attention
arithmetic.  Both the CUDA path (tests, bench, smoke) and the CPU oracle take
their inputs from here, so both sides see bit-identical bf16 values.

Recipe (the pages publish no dataset; these stand in for their workloads):
  * tensors Q, K, V, dO are [B, H, N, d], drawn on the CPU with
    ``torch.Generator().manual_seed(1000 * cfg + t)``, t = 0, 1, 2, 3 for
    Q, K, V, dO;
  * each is ``randn`` in fp32, multiplied by sigma, then rounded to bf16
    (round-to-nearest-even);
  * sigma = 1, except Q and K of the N=16384 workload, where sigma = 2 (a
    wide logit range that stresses the running-max rescale);
  * scale = 1/sqrt(d), computed in double and passed as fp32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    cfg: int
    B: int
    H: int
    N: int
    d: int
    causal: bool
    bwd: bool
    sigma_qk: float = 1.0

    @property
    def name(self) -> str:
        return (f"B{self.B}_H{self.H}_N{self.N}_d{self.d}_"
                f"{'causal' if self.causal else 'noncausal'}")

    @property
    def scale(self) -> float:
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32).item())

    def flops_fwd(self) -> float:
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def flops_bwd(self) -> float:
        return 2.5 * self.flops_fwd()


# The five attention workloads (B, H, N, d, causal, passes, sigma of Q/K).
WORKLOADS = {
    1: Workload(1, 1, 2, 256, 64, False, True),
    2: Workload(2, 2, 16, 1024, 128, True, True),
    3: Workload(3, 4, 32, 4096, 64, False, False),
    4: Workload(4, 1, 16, 8192, 128, True, True),
    5: Workload(5, 1, 8, 16384, 128, True, True, sigma_qk=2.0),
}


def seeded_bf16(shape, seed: int, sigma: float = 1.0, dtype=torch.bfloat16) -> torch.Tensor:
    """fp32 N(0, 1) from a CPU generator seeded with ``seed``, times sigma,
    rounded to ``dtype`` (bf16 unless asked for f16)."""
    g = torch.Generator().manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if sigma != 1.0:
        x = x * sigma
    return x.to(dtype)


def make_inputs(w: Workload, seed_base: int | None = None, with_grad: bool | None = None):
    """Q, K, V (and dO when the workload has a backward pass) on the CPU, bf16,
    contiguous [B, H, N, d]."""
    base = 1000 * w.cfg if seed_base is None else int(seed_base)
    shape = (w.B, w.H, w.N, w.d)
    q = seeded_bf16(shape, base + 0, w.sigma_qk)
    k = seeded_bf16(shape, base + 1, w.sigma_qk)
    v = seeded_bf16(shape, base + 2, 1.0)
    grad = w.bwd if with_grad is None else with_grad
    if grad:
        do = seeded_bf16(shape, base + 3, 1.0)
        return q, k, v, do
    return q, k, v


def custom(B: int, H: int, N: int, d: int, causal: bool, seed: int, sigma_qk: float = 1.0, dtype=torch.bfloat16):
    """Inputs for an ad-hoc shape (edge-case tests): Q, K, V, dO on the CPU,
    contiguous [B, H, N, d], bf16 (or f16)."""
    w = Workload(0, B, H, N, d, causal, True, sigma_qk)
    shape = (B, H, N, d)
    ins = tuple(seeded_bf16(shape, seed + t, sigma_qk if t < 2 else 1.0, dtype) for t in range(4))
    return w, ins

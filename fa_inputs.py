"""Seeded synthetic inputs for exact attention, shared by the tests, the bench and the oracle checks.

This module only draws random numbers and names workloads. It holds none of the attention
arithmetic: neither the CUDA path nor the oracle imports anything from the other through here.

Recipe (every workload): one CPU ``torch.Generator`` seeded with the workload's seed draws, in this
order, Q, K, V and (for the backward workloads) the upstream gradient dO, each as
``torch.randn(B, H, N, d, dtype=float32)``.  A workload with ``q_gain != 1`` multiplies Q by that gain in
fp32 (the peaky-row case).  bf16 workloads then round each tensor to bf16 (round to nearest even).
All tensors are contiguous ``[B, H, N, d]``.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str          # "f32" or "bf16": the element type the path reads and writes
    B: int
    H: int
    N: int
    d: int
    seed: int
    q_gain: float = 1.0
    backward: bool = False
    sampled_rows: int = 0   # >0: the oracle checks only this many seeded query rows per head

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def fwd_flops(self) -> float:
        """Algorithmic forward flops: the two N x N x d contractions, 4*B*H*N^2*d."""
        return 4.0 * self.B * self.H * self.N * self.N * self.d

    def bwd_flops(self) -> float:
        """Algorithmic backward flops: five N x N x d contractions, 10*B*H*N^2*d."""
        return 10.0 * self.B * self.H * self.N * self.N * self.d


WORKLOADS = {
    w.name: w
    for w in [
        Workload("fp32-fwd-B1-H1-N64-d16", "f32", 1, 1, 64, 16, seed=0),
        Workload("bf16-fwdbwd-B4-H16-N2048-d64", "bf16", 4, 16, 2048, 64, seed=1, backward=True),
        Workload("bf16-fwdbwd-B1-H16-N8192-d128", "bf16", 1, 16, 8192, 128, seed=2, backward=True),
        Workload("bf16-fwd-B1-H8-N32768-d128-q4", "bf16", 1, 8, 32768, 128, seed=3, q_gain=4.0),
        Workload("bf16-fwd-B1-H4-N131072-d128", "bf16", 1, 4, 131072, 128, seed=4, sampled_rows=256),
    ]
}

HEADLINE = "bf16-fwdbwd-B1-H16-N8192-d128"


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def make_inputs(B: int, H: int, N: int, d: int, dtype: str = "bf16", seed: int = 0,
                q_gain: float = 1.0, with_grad: bool = False) -> dict:
    """Draw q, k, v (and do when ``with_grad``) on the CPU as described in the module docstring."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    names = ["q", "k", "v"] + (["do"] if with_grad else [])
    out = {}
    for name in names:
        t = torch.randn(B, H, N, d, generator=g, dtype=torch.float32)
        if name == "q" and q_gain != 1.0:
            t.mul_(q_gain)
        out[name] = t.to(torch_dtype(dtype)).contiguous()
    return out


def workload_inputs(w: Workload, with_grad: bool | None = None) -> dict:
    return make_inputs(w.B, w.H, w.N, w.d, w.dtype, w.seed, w.q_gain,
                       w.backward if with_grad is None else with_grad)


def sample_rows(N: int, H: int, count: int = 256, seed_base: int = 1000) -> list:
    """Per head h, ``count`` distinct row indices drawn by ``randperm(N)`` under seed ``seed_base + h``, sorted."""
    rows = []
    for h in range(H):
        g = torch.Generator(device="cpu")
        g.manual_seed(seed_base + h)
        idx = torch.randperm(N, generator=g)[: min(count, N)]
        rows.append(torch.sort(idx).values)
    return rows

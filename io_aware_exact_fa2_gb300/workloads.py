"""Seeded synthetic inputs and the named workload shapes.

This module holds no attention arithmetic: it only draws random bf16 tensors
and names shapes.  Both the CUDA path's callers (tests, bench) and the fp64
oracle's callers take their inputs from here, so both sides see the same bytes.

Recipe (the pages benchmark on random tensors; there is no dataset):
  * Q, K, V are iid N(0, 1) drawn in fp32 from ``torch.Generator('cpu')``
    seeded with ``seed_base + {0, 1, 2}`` respectively, then rounded to bf16
    (round-to-nearest-even) on the CPU.
  * ``peaky_every = n`` multiplies every n-th key row (j % n == 0) by
    ``peaky_factor`` after the bf16 rounding; a factor that is a power of two
    is exact in bf16, so cast-then-scale equals scale-then-cast.
  * scale = 1 / sqrt(D).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Lq: int
    Lk: int
    D: int
    modes: tuple          # subset of ("noncausal", "causal")
    seed_base: int
    peaky_every: int = 0
    peaky_factor: float = 8.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def flops(self, causal: bool) -> float:
        """Attention forward FLOPs: 4*B*H*Lq*Lk*D, halved for causal."""
        f = 4.0 * self.B * self.H * self.Lq * self.Lk * self.D
        return f / 2.0 if causal else f

    def algorithmic_bytes(self) -> int:
        """Read Q, K, V once; write O (bf16) and LSE (fp32) once."""
        bh = self.B * self.H
        return bh * (2 * self.Lq * self.D * 2 + 2 * self.Lk * self.D * 2 + 4 * self.Lq)


# The five workloads: shapes, modes and seeds (seed_base = 1000 * index).
WORKLOADS = {
    "c1": Workload("c1", 1, 2, 128, 128, 64, ("noncausal", "causal"), 1000),
    "c2": Workload("c2", 4, 16, 1024, 1024, 64, ("noncausal", "causal"), 2000),
    "c3": Workload("c3", 2, 16, 4096, 4096, 128, ("noncausal", "causal"), 3000),
    "c4": Workload("c4", 1, 32, 16384, 16384, 128, ("causal",), 4000),
    "c5": Workload("c5", 2, 8, 2000, 3000, 256, ("noncausal",), 5000,
                   peaky_every=64, peaky_factor=8.0),
}


def randn_bf16(shape, seed: int) -> torch.Tensor:
    """iid N(0,1) fp32 from a seeded CPU generator, rounded to bf16."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randn(tuple(shape), generator=g, dtype=torch.float32).to(torch.bfloat16)


def make_qkv(B: int, H: int, Lq: int, Lk: int, D: int, seed_base: int,
             peaky_every: int = 0, peaky_factor: float = 8.0):
    """Seeded bf16 CPU tensors q (B,H,Lq,D), k and v (B,H,Lk,D)."""
    q = randn_bf16((B, H, Lq, D), seed_base + 0)
    k = randn_bf16((B, H, Lk, D), seed_base + 1)
    v = randn_bf16((B, H, Lk, D), seed_base + 2)
    if peaky_every:
        k[:, :, ::peaky_every, :] *= peaky_factor
    return q, k, v


def make_qkv_fp8(B: int, H: int, Lq: int, Lk: int, D: int, seed_base: int):
    """Seeded e4m3 (torch.float8_e4m3fn) q, k, v with fp32 descales of shape (B, H).

    The fp32 N(0, 1) draws are those of ``make_qkv`` (same seeds, before any bf16
    rounding).  Each (b, h) slice is divided by its descale = max|x| / 448 (e4m3's
    largest finite value; 1 for an all-zero slice) and cast to e4m3 (round to
    nearest even); the real input the pair stands for is stored value x descale.
    Returns (q8, k8, v8, dq, dk, dv), descales as float32 numpy arrays.
    """
    import numpy as np

    def quant(shape, seed):
        g = torch.Generator(device="cpu")
        g.manual_seed(int(seed))
        x = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
        amax = x.abs().amax(dim=(2, 3))
        ds = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
        return (x / ds[:, :, None, None]).to(torch.float8_e4m3fn), ds.numpy().astype(np.float32)

    q8, dq = quant((B, H, Lq, D), seed_base + 0)
    k8, dk = quant((B, H, Lk, D), seed_base + 1)
    v8, dv = quant((B, H, Lk, D), seed_base + 2)
    return q8, k8, v8, dq, dk, dv


def workload_inputs(w: Workload):
    return make_qkv(w.B, w.H, w.Lq, w.Lk, w.D, w.seed_base, w.peaky_every, w.peaky_factor)

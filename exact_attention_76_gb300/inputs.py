"""Seeded synthetic inputs shared by the tests, the bench and the CPU oracle.

This module only draws random numbers and rounds them to the storage types the
kernels read; it holds none of the attention arithmetic.  Both sides of every
parity check take their inputs from here and from nowhere else.

Recipe (the pages use no public dataset; these draws stand in for the training
shapes the pages discuss):
  * one ``torch.Generator('cpu')`` seeded with ``seed``;
  * draw order Q, K, V, dO; each i.i.d. N(0, 1) in fp32, shape [B, H, N, d];
  * bf16 storage by round-to-nearest-even (``Tensor.to(torch.bfloat16)``);
  * FP8 workloads: Q, K, V in fp32 with a Bernoulli(0.001) outlier mask per
    tensor whose entries are multiplied by 10; their e4m3 storage is made by
    the library's quantiser or, in the tests, by the oracle's (not here).

The named workloads are the training shapes the pages talk about: a tiny case,
a GPT-2-small-like layer, a sweep at fixed tokens, a long-context causal layer
and an FP8 forward.
"""
from __future__ import annotations

import dataclasses
import math

import torch

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int
    fp8: bool = False

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# The five workloads: tiny, GPT-2-small-like, fixed-token sweep, long causal, FP8.
TINY = Workload("tiny_B1_H2_N128_d64", 1, 2, 128, 64, False, 0)
GPT2 = Workload("gpt2small_B4_H12_N1024_d64", 4, 12, 1024, 64, True, 1)
LONG_CAUSAL = Workload("long_causal_B2_H16_N8192_d128", 2, 16, 8192, 128, True, 3)
FP8 = Workload("fp8_B1_H16_N16384_d128", 1, 16, 16384, 128, True, 4, fp8=True)


def sweep_workloads(causal: bool, d: int) -> list[Workload]:
    """Fixed 16384 tokens per batch, hidden 2048: H=32 at d=64, H=16 at d=128."""
    H = 2048 // d
    out = []
    for N in (512, 1024, 2048, 4096, 8192, 16384):
        out.append(Workload(f"sweep_B{16384 // N}_H{H}_N{N}_d{d}_{'c' if causal else 'nc'}",
                            16384 // N, H, N, d, causal, 2))
    return out


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def draw_fp32(B: int, H: int, N: int, d: int, seed: int):
    """Q, K, V, dO as fp32 N(0,1), drawn in that order from one generator."""
    g = _gen(seed)
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    do = torch.randn(shape, generator=g, dtype=torch.float32)
    return q, k, v, do


def draw_bf16(B: int, H: int, N: int, d: int, seed: int):
    """bf16 storage of :func:`draw_fp32` (round to nearest even)."""
    return tuple(t.to(torch.bfloat16) for t in draw_fp32(B, H, N, d, seed))


def draw_outlier_fp32(B: int, H: int, N: int, d: int, seed: int):
    """Q, K, V as N(0,1) with 0.1% of the entries of each tensor scaled by 10."""
    g = _gen(seed)
    shape = (B, H, N, d)
    out = []
    for _ in range(3):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        mask = torch.rand(shape, generator=g, dtype=torch.float32) < 1e-3
        x = torch.where(mask, x * 10.0, x)
        out.append(x)
    return tuple(out)


def make_bf16(w: Workload):
    return draw_bf16(w.B, w.H, w.N, w.d, w.seed)

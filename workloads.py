"""Seeded synthetic inputs for the BF16 GEMM, shared by the tests, the oracle
checks and the benchmark.

This module only draws numbers; it holds none of the product's arithmetic.
Every matrix is drawn in binary32 from a seeded ``torch.Generator`` on the CPU
and rounded to bfloat16 by torch's conversion (round to nearest even).  The
recipes mirror the workloads the pages talk about: decode-shaped linear layers
with K = 4096 (Llama-3-8B hidden size, Tencent AI-infra article, section
"演算子チューニング"), large square products, and long-K split-K problems.

Recipes (seed = 1234 + workload index unless a caller passes another):

====  ==============================================  ==========================
name  shapes                                          values
====  ==============================================  ==========================
small M=64,  N=256,  K=512                             A, B ~ N(0, 1)
decode M in {1,4,16,64}, N=4096, K=4096                A ~ N(0,1), B ~ N(0, 0.02)
square M=N=K in {2048, 4096, 8192}                     A, B ~ U(-1, 1)
large M=N=K=16384                                      A, B ~ N(0, 1)
longk M=N=256, K=65536                                 A, B ~ N(0, 1)
====  ==============================================  ==========================
"""
from __future__ import annotations

import torch

BASE_SEED = 1234

WORKLOADS = {
    "small": dict(index=0, M=64, N=256, K=512, dist="normal", a_std=1.0, b_std=1.0),
    "decode": dict(index=1, Ms=(1, 4, 16, 64), N=4096, K=4096, dist="normal",
                   a_std=1.0, b_std=0.02),
    "square": dict(index=2, sizes=(2048, 4096, 8192), dist="uniform"),
    "large": dict(index=3, M=16384, N=16384, K=16384, dist="normal", a_std=1.0, b_std=1.0),
    "longk": dict(index=4, M=256, N=256, K=65536, dist="normal", a_std=1.0, b_std=1.0,
                  splits=(8, 16, 32)),
}


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, seed: int, std: float = 1.0) -> torch.Tensor:
    g = generator(seed)
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def uniform_bf16(shape, seed: int, lo: float = -1.0, hi: float = 1.0) -> torch.Tensor:
    g = generator(seed)
    x = torch.rand(*shape, generator=g, dtype=torch.float32)
    x.mul_(hi - lo).add_(lo)
    return x.to(torch.bfloat16)


def int_bf16(shape, seed: int, lo: int = -8, hi: int = 8) -> torch.Tensor:
    """Small integers in [lo, hi] stored as bf16 (exact for |v| <= 256)."""
    g = generator(seed)
    x = torch.randint(lo, hi + 1, tuple(shape), generator=g, dtype=torch.int32)
    return x.to(torch.bfloat16)


def scaled_slices_bf16(shape, seed: int, scale_exp: int) -> torch.Tensor:
    """Entries n * 2^scale_exp with integer |n| <= 255 (at most 8 significant
    bits each, one shared power-of-two scale): the structure of the BF16
    slices in the cuTile/Ozaki article (techplay.jp, "最適化後の結果")."""
    g = generator(seed)
    n = torch.randint(-255, 256, tuple(shape), generator=g, dtype=torch.int32)
    x = n.to(torch.float32) * (2.0 ** scale_exp)
    return x.to(torch.bfloat16)


def pair(M: int, N: int, K: int, seed: int, dist: str = "normal",
         a_std: float = 1.0, b_std: float = 1.0):
    """(A [M,K], B [K,N]) bf16 CPU tensors for one GEMM."""
    if dist == "normal":
        return normal_bf16((M, K), seed, a_std), normal_bf16((K, N), seed + 7919, b_std)
    if dist == "uniform":
        return uniform_bf16((M, K), seed), uniform_bf16((K, N), seed + 7919)
    if dist == "int":
        return int_bf16((M, K), seed), int_bf16((K, N), seed + 7919)
    raise ValueError(dist)


def padded(t: torch.Tensor, ld: int) -> torch.Tensor:
    """Copy a 2-D tensor into a wider buffer (row stride ``ld``) and return the
    [rows, cols] view; the extra columns hold a NaN canary."""
    rows, cols = t.shape
    buf = torch.full((rows, ld), float("nan"), dtype=t.dtype)
    buf[:, :cols] = t
    return buf[:, :cols]

"""Seeded synthetic operands for the GEMM workloads.

This module only draws numbers: it holds none of the product's arithmetic,
and both the CUDA path and the oracle take their inputs from it.  Every
tensor is drawn on the CPU from a ``torch.Generator`` and rounded to f16
there (round to nearest even), so the GPU and the oracle see the same bits.

Distributions (the workload list below names one per operand pair):

* ``uniform``          -- U[-1, 1): ``rand * 2 - 1`` in f32, then f16.
* ``int4``             -- integers in [-4, 4], inclusive, stored as f16.
* ``normal``           -- N(0, 1).
* ``normal_invsqrtk``  -- N(0, 1) / sqrt(K), i.e. standard deviation 1/sqrt(K).
* ``ones``             -- all 1.0 (closed-form checks).

A is drawn before B from one generator seeded with the workload's seed.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

DISTRIBUTIONS = ("uniform", "int4", "normal", "normal_invsqrtk", "ones")


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dist: str
    seed: int
    batch: int = 1

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K * self.batch

    @property
    def algorithmic_bytes(self) -> int:
        """Read A and B once (f16), write C once (f32)."""
        return self.batch * (2 * self.M * self.K + 2 * self.K * self.N
                             + 4 * self.M * self.N)


# The five GEMM shapes, each with its operand distribution.  Seeds are
# 1000 + the shape's position; the small-integer twin of a shape uses +500.
WORKLOADS = {
    w.name: w
    for w in (
        Workload("gemm_64x128x128_uniform", 64, 128, 128, "uniform", 1000),
        Workload("gemm_64x128x128_int4", 64, 128, 128, "int4", 1500),
        Workload("gemm_1000x1000x1000_normal", 1000, 1000, 1000, "normal", 1001),
        Workload("gemm_4096x4096x4096_normal_invsqrtk", 4096, 4096, 4096,
                 "normal_invsqrtk", 1002),
        Workload("gemm_256x256x65536_uniform", 256, 256, 65536, "uniform", 1003),
        Workload("gemm_8192x8192x8192_normal_invsqrtk", 8192, 8192, 8192,
                 "normal_invsqrtk", 1004),
    )
}


def integer_twin(w: Workload) -> Workload:
    """The same shape with small-integer inputs in [-4, 4] (seed + 500)."""
    if w.dist == "int4":
        return w
    return Workload(w.name.rsplit("_", 1)[0] + "_int4", w.M, w.N, w.K, "int4",
                    w.seed + 500, w.batch)


def draw(shape, dist: str, gen: torch.Generator, K: int) -> torch.Tensor:
    """One f16 CPU tensor of ``shape`` from ``dist``."""
    if dist == "uniform":
        x = torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    elif dist == "int4":
        x = torch.randint(-4, 5, shape, generator=gen, dtype=torch.int32).float()
    elif dist == "normal":
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
    elif dist == "normal_invsqrtk":
        x = torch.randn(shape, generator=gen, dtype=torch.float32) / math.sqrt(max(K, 1))
    elif dist == "ones":
        x = torch.ones(shape, dtype=torch.float32)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return x.to(torch.float16)


def operands(M: int, N: int, K: int, dist: str, seed: int, batch: int = 1,
             lda: int | None = None, ldb: int | None = None,
             pad_value: float = float("nan")):
    """Draw A (batch x M x K) and B (batch x K x N) as f16 CPU tensors.

    With ``lda > K`` (or ``ldb > N``) the operand is returned as a strided
    view into a wider buffer whose extra columns hold ``pad_value`` (NaN by
    default), so a kernel that read past the logical edge would be caught.
    The batch dimension is dropped when ``batch == 1``."""
    gen = torch.Generator().manual_seed(int(seed))
    a = draw((batch, M, K), dist, gen, K)
    b = draw((batch, K, N), dist, gen, K)
    if lda is not None and lda != K:
        if lda < K:
            raise ValueError("lda < K")
        buf = torch.full((batch, M, lda), pad_value, dtype=torch.float16)
        buf[:, :, :K] = a
        a = buf[:, :, :K]
    if ldb is not None and ldb != N:
        if ldb < N:
            raise ValueError("ldb < N")
        buf = torch.full((batch, K, ldb), pad_value, dtype=torch.float16)
        buf[:, :, :N] = b
        b = buf[:, :, :N]
    if batch == 1:
        a, b = a[0], b[0]
    return a, b


def workload_operands(w: Workload, **kw):
    return operands(w.M, w.N, w.K, w.dist, w.seed, w.batch, **kw)

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


# ------------------------------------------------------------------ grouped

@dataclass(frozen=True)
class GroupedWorkload:
    """A Mixture-of-Experts shape: ``groups`` experts, each with room for M
    token rows; ``tokens`` routed token slots are spread over the experts by
    ``group_counts`` (so each expert's row count is known only once drawn)."""
    name: str
    groups: int
    M: int
    N: int
    K: int
    tokens: int
    dist: str
    seed: int

    def counts(self) -> torch.Tensor:
        return group_counts(self.groups, self.M, self.tokens, self.seed)

    def flops(self, counts=None) -> int:
        c = self.counts() if counts is None else counts
        return 2 * int(c.sum()) * self.N * self.K

    def algorithmic_bytes(self, counts=None) -> int:
        """The used rows of A once (f16), every expert's B once (f16), the
        used rows of C once (f32)."""
        rows = int((self.counts() if counts is None else counts).sum())
        return 2 * rows * self.K + 2 * self.groups * self.K * self.N + 4 * rows * self.N


def group_counts(groups: int, M: int, tokens: int, seed: int) -> torch.Tensor:
    """Row counts of a routed batch (int32, CPU): every token slot picks an
    expert at random, expert e with probability softmax(z)[e] for z ~ N(0, 1)
    drawn once (some experts popular, some nearly idle); an expert keeps at
    most M slots (the rest are dropped, as a capacity limit does)."""
    gen = torch.Generator().manual_seed(int(seed) + 7)
    z = torch.randn(groups, generator=gen, dtype=torch.float64)
    probs = torch.softmax(z, dim=0)
    picks = torch.multinomial(probs, tokens, replacement=True, generator=gen)
    counts = torch.bincount(picks, minlength=groups).clamp(max=M)
    return counts.to(torch.int32)


def grouped_operands(w: GroupedWorkload):
    """A (groups x M x K) and B (groups x K x N) f16 CPU tensors: A drawn
    first, then B, from one generator seeded with the workload's seed."""
    gen = torch.Generator().manual_seed(int(w.seed))
    a = draw((w.groups, w.M, w.K), w.dist, gen, w.K)
    b = draw((w.groups, w.K, w.N), w.dist, gen, w.K)
    return a, b


# Two expert layouts, rows drawn from N(0, 1/sqrt(K)): a few wide experts
# (8 experts of 4096 x 14336, 16384 routed slots = 8192 tokens x top-2) and
# many narrow ones (64 experts of 2048 x 1408, 24576 slots = 4096 tokens x
# top-6), each expert with room for M rows.
GROUPED_WORKLOADS = {
    w.name: w
    for w in (
        GroupedWorkload("moe_8x4096x14336x4096_normal_invsqrtk", 8, 4096, 14336, 4096, 16384,
                        "normal_invsqrtk", 2000),
        GroupedWorkload("moe_64x512x1408x2048_normal_invsqrtk", 64, 512, 1408, 2048, 24576,
                        "normal_invsqrtk", 2001),
    )
}


# ------------------------------------------------------------------ row reductions

@dataclass(frozen=True)
class RowReduceWorkload:
    """A row sum (out[r] = sum_c x[r, c]) of an R x C matrix of `elem`
    values, or a GEMV (y = A x, A R x C f16) -- memory-bound: every element is
    read once.  Values U[-1, 1) drawn like the GEMM operands."""
    name: str
    kind: str   # "rowsum" or "gemv"
    R: int
    C: int
    elem: str   # "f32", "f16" or "bf16" (the GEMV is f16)
    seed: int

    @property
    def flops(self) -> int:
        return (2 if self.kind == "gemv" else 1) * self.R * self.C

    @property
    def algorithmic_bytes(self) -> int:
        eb = 4 if self.elem == "f32" else 2
        return self.R * self.C * eb + 4 * self.R + (2 * self.C if self.kind == "gemv" else 0)

    def operands(self):
        """(X or A as an R x C CPU tensor, x or None)."""
        gen = torch.Generator().manual_seed(int(self.seed))
        dt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[self.elem]
        X = (torch.rand((self.R, self.C), generator=gen, dtype=torch.float32) * 2.0 - 1.0).to(dt)
        x = None
        if self.kind == "gemv":
            x = (torch.rand(self.C, generator=gen, dtype=torch.float32) * 2.0 - 1.0).to(torch.float16)
        return X, x


# Sizes above the L2 (every element comes from HBM): many medium rows, a few
# very long rows (cut into segments), and the f16 GEMV.
ROW_WORKLOADS = {
    w.name: w
    for w in (
        RowReduceWorkload("rowsum_8192x32768_f16", "rowsum", 8192, 32768, "f16", 3000),
        RowReduceWorkload("rowsum_4x33554432_f32", "rowsum", 4, 33554432, "f32", 3001),
        RowReduceWorkload("rowsum_262144x1024_bf16", "rowsum", 262144, 1024, "bf16", 3002),
        RowReduceWorkload("gemv_16384x16384_f16", "gemv", 16384, 16384, "f16", 3003),
    )
}

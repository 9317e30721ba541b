"""Helpers for the GPU parity tests: padded device operands with NaN guard
bands, a sentinel-filled output, and the tolerance of the f32 result."""
from __future__ import annotations

import math

import numpy as np
import torch

SENTINEL = 1.0e30  # C's row padding and guard band must keep this value
GUARD = 256        # elements after each buffer


class DeviceMatrix:
    """``batch`` row-major matrices in one flat device buffer, row stride
    ``ld``, batch stride ``stride``; everything outside the logical
    ``rows x cols`` blocks (row padding, gaps between batches, a guard band
    after the end) holds ``fill``."""

    def __init__(self, x: torch.Tensor | None, rows: int, cols: int, ld: int, dtype,
                 fill: float, batch: int = 1, stride: int | None = None,
                 inner_fill: float | None = None):
        self.rows, self.cols, self.ld, self.batch = rows, cols, ld, batch
        self.stride = stride if stride is not None else rows * ld
        total = (batch - 1) * self.stride + rows * ld + GUARD
        self.buf = torch.full((total,), fill, dtype=dtype, device="cuda")
        self.fill = fill
        if inner_fill is not None:
            for b in range(batch):
                self.block(b)[:, :cols] = inner_fill
        if x is not None:
            xs = x.reshape(batch, rows, cols)
            for b in range(batch):
                self.block(b)[:, :cols] = xs[b].to(device="cuda", dtype=dtype)

    def block(self, b: int = 0) -> torch.Tensor:
        o = b * self.stride
        return self.buf[o:o + self.rows * self.ld].view(self.rows, self.ld)

    def ptr(self) -> int:
        return self.buf.data_ptr()

    def logical(self) -> torch.Tensor:
        """The logical matrices, copied to the CPU (batch x rows x cols)."""
        return torch.stack([self.block(b)[:, :self.cols] for b in range(self.batch)]).cpu()

    def outside_untouched(self) -> bool:
        mask = torch.ones(self.buf.numel(), dtype=torch.bool, device="cuda")
        for b in range(self.batch):
            o = b * self.stride
            m = mask[o:o + self.rows * self.ld].view(self.rows, self.ld)
            m[:, :self.cols] = False
        outside = self.buf[mask]
        if math.isnan(self.fill):
            return bool(torch.isnan(outside).all())
        return bool((outside == self.fill).all())


def run_gemm(b, A: torch.Tensor, B: torch.Tensor, *, lda=None, ldb=None, ldc=None, batch=1,
             sA=None, sB=None, sC=None, split_k=0, tile_n=0, tile_m=0, splitk_reduce=0,
             split_tail=0, red_cluster=0, stream=None):
    """A: (batch,) M x K f16 CPU, B: (batch,) K x N f16 CPU.  Runs the GEMM
    through the C ABI on padded device buffers and returns (C as a CPU f32
    tensor of shape (batch,) M x N, the output DeviceMatrix)."""
    M, K = A.shape[-2], A.shape[-1]
    N = B.shape[-1]
    lda = lda or max(8, -(-K // 8) * 8)
    ldb = ldb or max(8, -(-N // 8) * 8)
    ldc = ldc or max(4, -(-N // 4) * 4)
    dA = DeviceMatrix(A, M, K, lda, torch.float16, float("nan"), batch, sA)
    dB = DeviceMatrix(B, K, N, ldb, torch.float16, float("nan"), batch, sB)
    dC = DeviceMatrix(None, M, N, ldc, torch.float32, SENTINEL, batch, sC,
                      inner_fill=float("nan"))
    opts = b.GemmOptions(split_k, tile_n, 0, 0, tile_m, splitk_reduce, 0, split_tail)
    opts.red_cluster = red_cluster
    s = torch.cuda.current_stream() if stream is None else stream
    st = b.gemm_f16_f32acc_opts(dA.ptr(), dB.ptr(), dC.ptr(), M, N, K, lda, ldb, ldc,
                                dA.stride if batch > 1 else 0, dB.stride if batch > 1 else 0,
                                dC.stride if batch > 1 else 0, batch, opts, s.cuda_stream)
    b.check(st)
    b.check(b.gemm_get_device_status(s.cuda_stream))
    C = dC.logical()
    return (C if batch > 1 else C[0]), dC


def check_tolerance(C: np.ndarray, ref: np.ndarray, K: int) -> dict:
    """The f32 result against the fp64 oracle: finite everywhere,
    max |C - ref| <= 1e-3 sqrt(K), relative Frobenius error <= 1e-4."""
    C = np.asarray(C, dtype=np.float64)
    assert np.all(np.isfinite(C)), "non-finite output"
    err = np.abs(C - ref)
    max_err = float(err.max()) if err.size else 0.0
    denom = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(C - ref) / denom) if denom > 0 else float(np.linalg.norm(C - ref))
    assert max_err <= 1e-3 * math.sqrt(max(K, 1)), f"max abs error {max_err}"
    assert rel <= 1e-4, f"relative Frobenius error {rel}"
    return {"max_abs": max_err, "rel_fro": rel}


def check_exact(C: np.ndarray, ref: np.ndarray) -> None:
    C = np.asarray(C, dtype=np.float32)
    R = ref.astype(np.float32)
    assert np.array_equal(R.astype(np.float64), ref), "reference not exact in f32"
    bad = np.argwhere(C != R)
    assert bad.size == 0, f"{len(bad)} cells differ, first {bad[:3].tolist()}"

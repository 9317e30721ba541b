"""Operands the tensor-memory accelerator cannot address, on the GPU.

Bases that are not 16-byte aligned and row or batch pitches that are not
multiples of 16 bytes go through a packed, aligned copy (C is computed there
and copied out).  Each case lays its operands out at such offsets and
pitches in NaN-filled buffers, surrounds C with a sentinel, and compares
with the oracle: bit for bit on small-integer inputs, within the tolerance
on random ones; everything outside C's logical blocks (and, in a grouped
call, C's rows past each count) must keep its value."""
import numpy as np
import pytest
import torch

import oracle
from tiled_staged_matmul_gb300 import synthetic

from gpu_util import SENTINEL, check_exact, check_tolerance

pytestmark = pytest.mark.gpu

GUARD = 64


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.fail("the GPU tests need a CUDA device")
    from tiled_staged_matmul_gb300 import binding
    return binding


class Strided:
    """`batch` matrices of rows x cols at element `offset` of a flat buffer,
    row pitch `ld`, batch pitch `stride`; the rest of the buffer holds `fill`."""

    def __init__(self, x, rows, cols, ld, stride, offset, dtype, fill, inner=None):
        self.rows, self.cols, self.ld, self.stride, self.offset = rows, cols, ld, stride, offset
        self.batch = 1 if x is None and inner is None else None
        batch = x.shape[0] if x is not None else inner
        self.batch = batch
        total = offset + (batch - 1) * stride + rows * ld + GUARD
        self.buf = torch.full((total,), fill, dtype=dtype, device="cuda")
        self.fill = fill
        for i in range(batch):
            blk = self.block(i)
            if x is not None:
                blk[:, :cols] = x[i].to(device="cuda", dtype=dtype)

    def block(self, i):
        o = self.offset + i * self.stride
        return self.buf[o:o + self.rows * self.ld].view(self.rows, self.ld)

    def ptr(self):
        return self.buf.data_ptr() + self.offset * self.buf.element_size()

    def logical(self):
        return torch.stack([self.block(i)[:, :self.cols] for i in range(self.batch)]).cpu()

    def outside_is_fill(self):
        mask = torch.ones(self.buf.numel(), dtype=torch.bool, device="cuda")
        for i in range(self.batch):
            o = self.offset + i * self.stride
            mask[o:o + self.rows * self.ld].view(self.rows, self.ld)[:, :self.cols] = False
        rest = self.buf[mask]
        return bool(torch.isnan(rest).all()) if np.isnan(self.fill) else bool((rest == self.fill).all())


def layout(M, N, K, batch, lda, ldb, ldc, offs=(0, 0, 0), extra=(0, 0, 0)):
    sA = M * lda + extra[0]
    sB = K * ldb + extra[1]
    sC = M * ldc + extra[2]
    return dict(lda=lda, ldb=ldb, ldc=ldc, sA=sA, sB=sB, sC=sC, offs=offs)


def run_case(b, A, B, L, opts=None):
    batch, M, K = A.shape
    N = B.shape[2]
    dA = Strided(A, M, K, L["lda"], L["sA"], L["offs"][0], torch.float16, float("nan"))
    dB = Strided(B, K, N, L["ldb"], L["sB"], L["offs"][1], torch.float16, float("nan"))
    dC = Strided(None, M, N, L["ldc"], L["sC"], L["offs"][2], torch.float32, SENTINEL, inner=batch)
    s = torch.cuda.current_stream().cuda_stream
    b.check(b.gemm_f16_f32acc_opts(dA.ptr(), dB.ptr(), dC.ptr(), M, N, K, L["lda"], L["ldb"], L["ldc"],
                                   L["sA"] if batch > 1 else 0, L["sB"] if batch > 1 else 0,
                                   L["sC"] if batch > 1 else 0, batch, opts, s))
    b.check(b.gemm_get_device_status(s))
    C = dC.logical().double().numpy()
    # C's padding holds the sentinel except inside the logical blocks
    mask_ok = dC.outside_is_fill()
    return C, mask_ok


def refs(A, B):
    batch, M, K = A.shape
    N = B.shape[2]
    return np.stack([oracle.gemm_f64(A[i].contiguous(), B[i].contiguous(), M, N, K) for i in range(batch)])


CASES = {
    "odd lda": (1, 300, 200, 520, dict(lda=521, ldb=200, ldc=200)),
    "odd ldb": (1, 300, 203, 520, dict(lda=520, ldb=205, ldc=204)),
    "odd ldc": (1, 300, 201, 520, dict(lda=520, ldb=208, ldc=201)),
    "unaligned bases": (1, 257, 136, 264, dict(lda=264, ldb=136, ldc=136, offs=(1, 3, 1))),
    "batched odd strides": (3, 130, 70, 200, dict(lda=203, ldb=70, ldc=71, extra=(5, 1, 2))),
    "everything odd": (2, 65, 33, 95, dict(lda=97, ldb=35, ldc=37, offs=(3, 5, 3), extra=(1, 3, 1))),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_unaddressable_layouts_are_exact(b, name):
    batch, M, N, K, kw = CASES[name]
    A, B = synthetic.operands(M, N, K, "int4", seed=60 + sorted(CASES).index(name), batch=batch)
    if batch == 1:
        A, B = A[None], B[None]
    L = layout(M, N, K, batch, kw["lda"], kw["ldb"], kw["ldc"], kw.get("offs", (0, 0, 0)),
               kw.get("extra", (0, 0, 0)))
    C, outside_ok = run_case(b, A, B, L)
    check_exact(C, refs(A, B))
    assert outside_ok


@pytest.mark.parametrize("tile_m,tile_n", [(128, 64), (256, 256)])
def test_unaddressable_layouts_random_inputs(b, tile_m, tile_n):
    M, N, K = 520, 330, 777
    A, B = synthetic.operands(M, N, K, "uniform", seed=51)
    L = layout(M, N, K, 1, 779, 333, 331, offs=(1, 1, 1))
    C, outside_ok = run_case(b, A[None], B[None], L, b.GemmOptions(0, tile_n, 0, 0, tile_m))
    check_tolerance(C[0], refs(A[None], B[None])[0], K)
    assert outside_ok


def test_long_K_split_through_the_repacked_operand(b):
    M, N, K = 256, 256, 16384
    A, B = synthetic.operands(M, N, K, "int4", seed=52)
    L = layout(M, N, K, 1, K + 4, N, N)     # lda not a multiple of 8: A repacked, K split
    assert b.gemm_plan(M, N, K, 1, None)["split_k"] > 1
    C, outside_ok = run_case(b, A[None], B[None], L)
    check_exact(C, refs(A[None], B[None]))
    assert outside_ok


def test_K_zero_with_unaligned_C_needs_no_copy(b):
    M, N = 40, 30
    dC = Strided(None, M, N, 31, M * 31, 1, torch.float32, SENTINEL, inner=1)
    b.check(b.gemm_f16_f32acc(0, 0, dC.ptr(), M, N, 0, 8, 8, 31, 0))
    b.check(b.gemm_get_device_status(0))
    assert bool((dC.logical() == 0).all()) and dC.outside_is_fill()


def test_grouped_copy_out_keeps_rows_past_each_count(b):
    G, M, N, K = 4, 200, 130, 72
    rows = [200, 0, 57, 129]
    A, B = synthetic.operands(M, N, K, "int4", seed=53, batch=G)
    prior = 7.5
    dA = Strided(A, M, K, K, M * K, 0, torch.float16, float("nan"))
    dB = Strided(B, K, N, 136, K * 136, 0, torch.float16, float("nan"))
    dC = Strided(None, M, N, 131, M * 131 + 1, 1, torch.float32, SENTINEL, inner=G)
    for g in range(G):
        dC.block(g)[:, :N] = prior
    counts = torch.tensor(rows, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    b.check(b.gemm_f16_f32acc_grouped(dA.ptr(), dB.ptr(), dC.ptr(), counts.data_ptr(), G, M, N, K,
                                      K, 136, 131, M * K, K * 136, M * 131 + 1, s))
    b.check(b.gemm_get_device_status(s))
    C = dC.logical().double().numpy()
    ref = oracle.grouped_gemm_f64(A, B, rows, G, M, N, K, C=np.full((G, M, N), prior))
    assert np.array_equal(C, ref)
    assert dC.outside_is_fill()


def test_noalloc_entry_refuses_unaddressable_layouts(b):
    M, N, K = 64, 64, 64
    A = torch.zeros(M * 72, dtype=torch.float16, device="cuda")
    B = torch.zeros(K * N, dtype=torch.float16, device="cuda")
    C = torch.zeros(M * N, dtype=torch.float32, device="cuda")
    st = b.gemm_f16_f32acc_splitk_noalloc(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, 70, N, N,
                                          0, 0)
    assert b.gemm_status_string(st) == "GEMM_ERR_MISALIGNED"


def test_benchmarked_odd_pitches_full_size(b, full_8192):
    """The bench's repacked line at full size: 8192^3 with every row pitch
    odd (A, B and C all repacked), every cell against the oracle; C's padding
    is left untouched."""
    from gpu_util import run_gemm
    w, A, B, ref = full_8192
    C, dC = run_gemm(b, A, B, lda=w.K + 1, ldb=w.N + 1, ldc=w.N + 1)
    check_tolerance(C.numpy(), ref, w.K)
    assert dC.outside_untouched()

"""Operands the tensor-memory accelerator cannot address, on the GPU.

Bases that are not 16-byte aligned and row or batch pitches that are not
multiples of 16 bytes go through a packed, aligned copy (C is computed there
and copied out).  Each case lays its operands out at such
offsets and pitches in NaN-filled buffers, surrounds C with a sentinel, and
compares with the oracle: bit for bit on small-integer inputs, within the
tolerance on random ones; everything outside C's logical blocks (and, in a
grouped call, C's rows past each count) must keep its value."""
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


def _opts(b, **kw):
    o = b.GemmOptions()
    for k, v in kw.items():
        setattr(o, k, v)
    return o


# A C the TMA cannot store to (odd ldc, C one element past a 16-byte
# boundary) under every plan that writes C: whole tiles, the separate reduce
# kernel, the end-of-launch in-kernel split-K sum, the CTA-pair split tail
# summed first (split units first), and the cluster sums.
ODD_C_PLANS = {
    "whole tiles": ((600, 330, 520), dict(split_k=1, split_tail=2), (1, 0)),
    "separate reduce": ((256, 130, 8192), dict(split_k=4, splitk_reduce=1), (1, 0)),
    "in-kernel sum": ((256, 130, 8192), dict(split_k=8, tile_m=128, tile_n=128), (1, 1)),
    "pair split tail": ((2304, 2304, 1024), dict(split_tail=1, tile_m=256, tile_n=256), (1, 1)),
    "cluster of 4": ((256, 256, 16384), dict(split_k=8, tile_m=128, tile_n=128, red_cluster=4), (4, 1)),
    "cluster of 2": ((200, 300, 20000), dict(split_k=12, tile_m=128, tile_n=128, red_cluster=2), (2, 1)),
}


@pytest.mark.parametrize("name", sorted(ODD_C_PLANS))
def test_odd_C_through_every_store_path(b, name):
    (M, N, K), fields, (want_cluster, want_fused) = ODD_C_PLANS[name]
    o = _opts(b, **fields)
    p = b.gemm_plan(M, N, K, 1, o)
    assert p["red_cluster"] == want_cluster and p["fused_reduce"] == want_fused, p
    if name == "pair split tail":
        assert p["tile_m"] == 256 and p["tail_split"] >= 2 and not p["tail_narrow"], p
    A, B = synthetic.operands(M, N, K, "int4", seed=M + N + K)
    L = layout(M, N, K, 1, K, N, N + 1, offs=(0, 0, 1))
    C, outside_ok = run_case(b, A[None], B[None], L, o)
    check_exact(C, refs(A[None], B[None]))
    assert outside_ok


@pytest.mark.parametrize("out", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("fields", [dict(split_tail=1, tile_m=256, tile_n=256),
                                    dict(split_k=8, tile_m=128, tile_n=128)])
def test_odd_C_with_the_fused_epilogue(b, out, fields):
    """16-bit and f32 outputs with an odd pitch through the split-K sums."""
    from test_epilogue_gpu import check_epilogue
    M, N, K = (2304, 2304, 1024) if "split_tail" in fields else (256, 130, 8192)
    A, B = synthetic.operands(M, N, K, "uniform", seed=K + 7)
    dA, dB = A.cuda().contiguous(), B.cuda().contiguous()
    dt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[out]
    ldc = N + 1
    fill = SENTINEL if out == "f32" else 1000.0
    buf = torch.full((1 + M * ldc + GUARD,), fill, dtype=dt, device="cuda")
    bias = torch.linspace(-1, 1, N, dtype=torch.float32, device="cuda")
    epi = b.epilogue(0.5, bias.data_ptr(), 0, "gelu", 0.01, out)
    s = torch.cuda.current_stream().cuda_stream
    b.check(b.gemm_f16_fused(dA.data_ptr(), dB.data_ptr(), buf.data_ptr() + buf.element_size(), M, N, K,
                             K, N, ldc, 0, 0, 0, 1, epi, _opts(b, **fields), s))
    b.check(b.gemm_get_device_status(s))
    C = buf[1:1 + M * ldc].view(M, ldc)
    check_epilogue(C[:, :N].float().cpu().double().numpy(), oracle.gemm_f64(A, B, M, N, K), 0.5,
                   bias.cpu().double().numpy(), "gelu", out, K)
    assert bool((C[:, N:] == fill).all()) and bool((buf[0] == fill).all())
    assert bool((buf[1 + M * ldc:] == fill).all())


def test_odd_C_grouped(b):
    G, M, N, K = 4, 300, 256, 512
    rows = [300, 0, 129, 17]
    A, B = synthetic.operands(M, N, K, "int4", seed=47, batch=G)
    ldc = N + 3
    dC = Strided(None, M, N, ldc, M * ldc + 1, 1, torch.float32, SENTINEL, inner=G)
    counts = torch.tensor(rows, dtype=torch.int32, device="cuda")
    dA, dB = A.cuda().contiguous(), B.cuda().contiguous()
    s = torch.cuda.current_stream().cuda_stream
    b.check(b.gemm_f16_f32acc_grouped(dA.data_ptr(), dB.data_ptr(), dC.ptr(), counts.data_ptr(), G, M, N,
                                      K, K, N, ldc, M * K, K * N, M * ldc + 1, s))
    b.check(b.gemm_get_device_status(s))
    C = dC.logical().double().numpy()
    for g in range(G):
        r = rows[g]
        ref = oracle.gemm_f64(A[g, :r].contiguous(), B[g], r, N, K) if r else np.zeros((0, N))
        assert np.array_equal(C[g, :r], ref)
        assert np.all(C[g, r:] == np.float32(SENTINEL))

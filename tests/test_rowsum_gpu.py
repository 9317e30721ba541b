"""The tiled row sum and the GEMV on the GPU against their oracles.

Row sums run on f32, f16 and bf16 views with every layout the call takes:
contiguous rows (the 16-byte vector path), padded and odd row strides, a
column stride (a transposed view sums columns), an unaligned base (the
element path), few long rows (cut into segments summed in a second pass)
and many short ones; the four benchmarked row workloads run at full size,
checked on sampled rows.  Bound: max |out - ref| <= 1e-3 sqrt(C) and relative
error <= 1e-4 (the GEMM's, with K = C); small-integer inputs must match
bit for bit, and repeated calls must agree bit for bit."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "row_sum_worked_examples.json")
TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.fail("the GPU tests need a CUDA device")
    from tiled_staged_matmul_gb300 import binding
    return binding


def bits_of(t):
    """The CPU buffer the oracle reads (f32 values or 16-bit patterns)."""
    t = t.detach().cpu().contiguous().reshape(-1)
    return t.numpy() if t.dtype == torch.float32 else t.view(torch.int16).numpy().view(np.uint16)


def check(out, ref, C, exact=False):
    out = np.asarray(out, dtype=np.float64)
    if exact:
        assert np.array_equal(out, ref.astype(np.float32).astype(np.float64))
        return
    assert np.all(np.isfinite(out))
    err = np.abs(out - ref)
    assert err.max(initial=0) <= 1e-3 * math.sqrt(max(C, 1)), err.max()
    denom = np.linalg.norm(ref)
    if denom > 0:
        assert np.linalg.norm(out - ref) / denom <= 1e-4


def run(b, buf, elem, R, C, rs, cs, offset=0):
    """Row sums of the view of `buf` (a flat CUDA tensor) at `offset`."""
    out = torch.full((R + 8,), float("nan"), dtype=torch.float32, device="cuda")
    ptr = buf.data_ptr() + offset * buf.element_size()
    b.check(b.rowsum_f32acc(ptr, elem, out.data_ptr(), R, C, rs, cs, 0))
    b.check(b.gemm_get_device_status(0))
    assert bool(torch.isnan(out[R:]).all()), "wrote past out"
    return out[:R].cpu().double().numpy()


def test_worked_values_from_the_page(b):
    for case in json.load(open(GOLDEN))["row_sums"]:
        x = torch.tensor(case["x"], dtype=torch.float32)
        R, C = x.shape
        for elem in ("f32", "f16", "bf16"):
            buf = x.to(TORCH[elem]).reshape(-1).cuda()
            assert run(b, buf, elem, R, C, C, 1).tolist() == case["expected"], (case["cite"], elem)


LAYOUTS = [
    # (R, C, row_stride, col_stride, offset): contiguous, padded, odd, strided,
    # transposed (row stride 1), unaligned base, few long rows, many short ones
    (1000, 1000, 1000, 1, 0),
    (257, 300, 312, 1, 0),
    (129, 301, 303, 1, 0),
    (64, 500, 1500, 3, 0),
    (300, 200, 1, 300, 0),
    (90, 777, 777, 1, 1),
    (3, 200003, 200003, 1, 0),
    (1, 1000000, 1000000, 1, 0),
    (50000, 7, 7, 1, 0),
    (20000, 3, 3, 1, 0),
    (7, 0, 5, 1, 0),
]


@pytest.mark.parametrize("elem", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("R,C,rs,cs,off", LAYOUTS)
def test_layouts_against_the_oracle(b, elem, R, C, rs, cs, off):
    size = off + (max(R, 1) - 1) * rs + (max(C, 1) - 1) * cs + 1
    gen = torch.Generator().manual_seed(R * 31 + C)
    vals = (torch.rand(size, generator=gen) * 2 - 1)
    buf = vals.to(TORCH[elem]).cuda()
    got = run(b, buf, elem, R, C, rs, cs, off)
    ref = oracle.rowsum_f64(bits_of(buf)[off:], R, C, rs, cs, elem)
    check(got, ref, C)


@pytest.mark.parametrize("elem", ["f32", "f16", "bf16"])
def test_integer_inputs_are_exact_and_calls_reproducible(b, elem):
    R, C = 333, 40000
    gen = torch.Generator().manual_seed(5)
    buf = torch.randint(-4, 5, (R * C,), generator=gen).to(TORCH[elem]).cuda()
    got = run(b, buf, elem, R, C, C, 1)
    check(got, oracle.rowsum_f64(bits_of(buf), R, C, C, 1, elem), C, exact=True)
    vals = (torch.rand(7 * 300001, generator=gen) * 2 - 1).to(TORCH[elem]).cuda()
    first = run(b, vals, elem, 7, 300001, 300001, 1)
    for _ in range(3):
        assert np.array_equal(run(b, vals, elem, 7, 300001, 300001, 1), first)


def test_torch_wrapper_on_views(b):
    x = (torch.rand(500, 600) * 2 - 1).half().cuda()
    for view in (x, x[:, 7:], x.t(), x[::3, ::2]):
        got = b.rowsum(view).cpu().double().numpy()
        ref = oracle.rowsum_f64(bits_of(view.contiguous()), view.shape[0], view.shape[1],
                                view.shape[1], 1, "f16")
        check(got, ref, view.shape[1])


@pytest.mark.parametrize("M,K,lda,incx,xoff", [
    (1000, 1000, 1000, 1, 0),
    (4096, 4096, 4096, 1, 0),
    (333, 777, 784, 1, 0),
    (300, 500, 501, 1, 0),
    (200, 300, 300, 3, 0),
    (100, 400, 400, 1, 1),
    (4, 262144, 262144, 1, 0),
    (50000, 9, 9, 1, 0),
    (12, 0, 8, 1, 0),
])
def test_gemv_against_the_oracle(b, M, K, lda, incx, xoff):
    gen = torch.Generator().manual_seed(M + K)
    A = (torch.rand(max(M * lda, 1), generator=gen) * 2 - 1).half().cuda()
    x = (torch.rand(xoff + max((K - 1) * incx + 1, 1), generator=gen) * 2 - 1).half().cuda()
    y = torch.full((M + 4,), float("nan"), dtype=torch.float32, device="cuda")
    b.check(b.gemv_f16_f32acc(A.data_ptr(), x.data_ptr() + 2 * xoff, y.data_ptr(), M, K, lda, incx, 0))
    b.check(b.gemm_get_device_status(0))
    assert bool(torch.isnan(y[M:]).all())
    ref = oracle.gemv_f64(bits_of(A).view(np.float16), bits_of(x)[xoff:].view(np.float16), M, K, lda, incx)
    check(y[:M].cpu().double().numpy(), ref, K)


def test_gemv_integer_exact_and_wrapper(b):
    gen = torch.Generator().manual_seed(9)
    A = torch.randint(-4, 5, (700, 3000), generator=gen).half().cuda()
    x = torch.randint(-4, 5, (3000,), generator=gen).half().cuda()
    y = b.gemv(A, x).cpu().double().numpy()
    ref = oracle.gemv_f64(bits_of(A).view(np.float16), bits_of(x).view(np.float16), 700, 3000)
    check(y, ref, 3000, exact=True)
    y2 = b.gemv(A[:, ::1], x[::1])
    assert np.array_equal(y2.cpu().double().numpy(), y)


@pytest.mark.parametrize("name", ["rowsum_8192x32768_f16", "rowsum_262144x1024_bf16",
                                  "rowsum_4x33554432_f32", "gemv_16384x16384_f16"])
def test_row_workloads_full_size_sampled(b, name):
    """The benchmarked row workloads at full size through the C ABI, checked
    against the oracle on sampled rows (all four of the long-row case)."""
    from tiled_staged_matmul_gb300 import synthetic
    w = synthetic.ROW_WORKLOADS[name]
    X, x = w.operands()
    dX = X.cuda()
    out = torch.full((w.R + 4,), float("nan"), dtype=torch.float32, device="cuda")
    if w.kind == "gemv":
        dx = x.cuda()
        b.check(b.gemv_f16_f32acc(dX.data_ptr(), dx.data_ptr(), out.data_ptr(), w.R, w.C, w.C, 1, 0))
    else:
        b.check(b.rowsum_f32acc(dX.data_ptr(), w.elem, out.data_ptr(), w.R, w.C, w.C, 1, 0))
    b.check(b.gemm_get_device_status(0))
    assert bool(torch.isnan(out[w.R:]).all()), "wrote past out"
    got = out[:w.R].cpu().double().numpy()
    rows = np.arange(w.R) if w.R <= 4 else np.unique(np.random.default_rng(5).integers(0, w.R, 64))
    Xs = X[torch.from_numpy(rows)].contiguous()
    if w.kind == "gemv":
        ref = oracle.gemv_f64(bits_of(Xs).view(np.float16), bits_of(x).view(np.float16), len(rows), w.C)
    else:
        ref = oracle.rowsum_f64(bits_of(Xs), len(rows), w.C, w.C, 1, w.elem)
    check(got[rows], ref, w.C)

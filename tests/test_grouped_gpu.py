"""Grouped (Mixture-of-Experts) GEMM on the GPU against the grouped oracle.

Each case runs through the C ABI on padded device buffers: NaN in A's and
B's padding, in A's rows at or past each group's count (loaded with the
tile that crosses the count, never allowed into C) and after every buffer;
C's rows below each count must match the oracle (bit for bit on
small-integer inputs, within max |C - C_ref| <= 1e-3 sqrt(K) and relative
Frobenius error <= 1e-4 on random ones), C's rows at or past the count must
keep their prior value, and everything outside C's logical blocks must keep
the sentinel."""
import numpy as np
import pytest
import torch

import oracle
from tiled_staged_matmul_gb300 import synthetic

from gpu_util import SENTINEL, DeviceMatrix, check_exact, check_tolerance

pytestmark = pytest.mark.gpu

PRIOR = 7.5  # C's rows at or past a group's count must keep this

TILES = [(128, 64), (128, 128), (128, 256), (256, 128), (256, 256), (256, 512)]


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.fail("the GPU tests need a CUDA device")
    from tiled_staged_matmul_gb300 import binding
    return binding


def _pad(n, m):
    return max(m, -(-n // m) * m)


def run_grouped(b, A, B, rows, *, tile_m=0, tile_n=0, check_status=True):
    """A: G x M x K f16 CPU, B: G x K x N f16 CPU, rows: G ints.  Returns
    (C as G x M x N float64, the output DeviceMatrix, the call's status)."""
    G, M, K = A.shape
    N = B.shape[2]
    lda, ldb, ldc = _pad(K, 8), _pad(N, 8), _pad(N, 4)
    dA = DeviceMatrix(A, M, K, lda, torch.float16, float("nan"), G)
    for g in range(G):
        r = min(max(int(rows[g]), 0), M)
        dA.block(g)[r:, :K] = float("nan")
    dB = DeviceMatrix(B, K, N, ldb, torch.float16, float("nan"), G)
    dC = DeviceMatrix(None, M, N, ldc, torch.float32, SENTINEL, G, inner_fill=PRIOR)
    counts = torch.tensor(list(rows), dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    opts = b.GemmOptions(0, tile_n, 0, 0, tile_m)
    b.check(b.gemm_f16_f32acc_grouped_opts(dA.ptr(), dB.ptr(), dC.ptr(), counts.data_ptr(), G, M, N,
                                           K, lda, ldb, ldc, dA.stride, dB.stride, dC.stride, opts,
                                           s))
    status = b.gemm_get_device_status(s)
    if check_status:
        b.check(status)
    return dC.logical().double().numpy(), dC, status


def reference(A, B, rows):
    G, M, K = A.shape
    N = B.shape[2]
    return oracle.grouped_gemm_f64(A.contiguous(), B.contiguous(), np.asarray(rows), G, M, N, K,
                                   C=np.full((G, M, N), PRIOR))


def compare(C, ref, rows, K, exact=False):
    for g, r in enumerate(rows):
        assert np.all(C[g, r:] == PRIOR), f"group {g}: rows past the count were written"
    used = np.concatenate([C[g, :r].reshape(-1) for g, r in enumerate(rows)] + [np.zeros(0)])
    want = np.concatenate([ref[g, :r].reshape(-1) for g, r in enumerate(rows)] + [np.zeros(0)])
    if used.size == 0:
        return
    if exact:
        check_exact(used, want)
    else:
        check_tolerance(used, want, K)


@pytest.mark.parametrize("tile_m,tile_n", TILES)
def test_ragged_counts_every_tile_shape(b, tile_m, tile_n):
    G, M, N, K = 7, 300, 200, 520
    rows = [0, 1, 128, 129, 300, 77, 256]
    A, B = synthetic.operands(M, N, K, "uniform", seed=31, batch=G)
    C, dC, _ = run_grouped(b, A, B, rows, tile_m=tile_m, tile_n=tile_n)
    compare(C, reference(A, B, rows), rows, K)
    assert dC.outside_untouched()


@pytest.mark.parametrize("tile_m,tile_n", [(128, 128), (256, 256), (256, 512)])
def test_integer_inputs_are_exact(b, tile_m, tile_n):
    G, M, N, K = 5, 257, 130, 96
    rows = [257, 3, 0, 200, 33]
    A, B = synthetic.operands(M, N, K, "int4", seed=32, batch=G)
    C, dC, _ = run_grouped(b, A, B, rows, tile_m=tile_m, tile_n=tile_n)
    compare(C, reference(A, B, rows), rows, K, exact=True)
    assert dC.outside_untouched()


def test_full_counts_equal_the_batched_call_bitwise(b):
    G, M, N, K = 3, 384, 256, 640
    A, B = synthetic.operands(M, N, K, "normal", seed=33, batch=G)
    C, _, _ = run_grouped(b, A, B, [M] * G, tile_m=128, tile_n=256)
    lda, ldb, ldc = K, N, N
    dA, dB = A.cuda().contiguous(), B.cuda().contiguous()
    dC = torch.empty((G, M, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    b.check(b.gemm_f16_f32acc_opts(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), M, N, K, lda, ldb,
                                   ldc, M * lda, K * ldb, M * ldc, G,
                                   b.GemmOptions(1, 256, 0, 0, 128), s))
    b.check(b.gemm_get_device_status(s))
    assert np.array_equal(C, dC.cpu().double().numpy())


def test_more_groups_than_one_launch_holds(b):
    G, M, N, K = 300, 40, 64, 64   # 256 + 44 groups: two launches
    rng = np.random.default_rng(34)
    rows = [int(x) for x in rng.integers(0, M + 1, size=G)]
    rows[255] = M
    rows[256] = 0
    A, B = synthetic.operands(M, N, K, "uniform", seed=34, batch=G)
    C, dC, _ = run_grouped(b, A, B, rows)
    compare(C, reference(A, B, rows), rows, K)
    assert dC.outside_untouched()


def test_all_groups_empty_and_K_zero(b):
    G, M, N, K = 4, 100, 36, 48
    A, B = synthetic.operands(M, N, K, "uniform", seed=35, batch=G)
    C, dC, _ = run_grouped(b, A, B, [0] * G)
    assert np.all(C == PRIOR) and dC.outside_untouched()
    # K == 0: the rows below each count are the empty sum, the rest untouched
    rows = [3, 0, 100, 51]
    A0 = torch.zeros((G, M, 0), dtype=torch.float16)
    B0 = torch.zeros((G, 0, N), dtype=torch.float16)
    C, dC, _ = run_grouped(b, A0, B0, rows)
    for g, r in enumerate(rows):
        assert np.all(C[g, :r] == 0.0) and np.all(C[g, r:] == PRIOR)
    assert dC.outside_untouched()


def test_counts_outside_range_are_clamped_and_reported(b):
    G, M, N, K = 3, 64, 32, 64
    rows = [M + 9, -4, 10]
    A, B = synthetic.operands(M, N, K, "int4", seed=36, batch=G)
    C, _, status = run_grouped(b, A, B, rows, check_status=False)
    assert b.gemm_status_string(status) == "GEMM_ERR_INVALID_VALUE"
    assert "row count" in b.gemm_last_error_string()
    clamped = [M, 0, 10]
    compare(C, reference(A, B, clamped), clamped, K, exact=True)
    assert b.gemm_get_device_status(0) == b.GEMM_OK  # reading the status cleared it


def test_counts_written_by_a_kernel_on_the_stream(b):
    """The counts are read when the GEMM runs: here a routing step on the
    same stream produces them just before the call."""
    G, M, N, K = 16, 160, 96, 128
    A, B = synthetic.operands(M, N, K, "uniform", seed=37, batch=G)
    gen = torch.Generator().manual_seed(37)
    picks = torch.randint(0, G, (1200,), generator=gen).cuda()
    counts = torch.bincount(picks, minlength=G).clamp(max=M).to(torch.int32)
    out = torch.full((G, M, N), PRIOR, dtype=torch.float32, device="cuda")
    from tiled_staged_matmul_gb300 import binding
    binding.grouped_gemm(A.cuda(), B.cuda(), counts, out=out)
    rows = counts.cpu().tolist()
    compare(out.cpu().double().numpy(), reference(A, B, rows), rows, K)


def test_torch_wrapper_zero_fills_unused_rows(b):
    G, M, N, K = 3, 50, 21, 24
    A, B = synthetic.operands(M, N, K, "int4", seed=38, batch=G, ldb=24)
    rows = [50, 0, 7]
    counts = torch.tensor(rows, dtype=torch.int32, device="cuda")
    Bd = torch.zeros((G, K, 24), dtype=torch.float16, device="cuda")
    Bd[:, :, :N] = B.cuda()
    out = b.grouped_gemm(A.cuda(), Bd[:, :, :N], counts)   # padded rows of B, ragged N
    C = out.cpu().double().numpy()
    ref = oracle.grouped_gemm_f64(A, B.contiguous(), rows, G, M, N, K, C=np.zeros((G, M, N)))
    assert np.array_equal(C, ref)
    # row stride 21: not TMA-addressable, served by repacking (out too: pitch 21)
    out = torch.full((G, M, N), PRIOR, dtype=torch.float32, device="cuda")
    b.grouped_gemm(A.cuda(), B.contiguous().cuda(), counts, out=out)
    ref = oracle.grouped_gemm_f64(A, B.contiguous(), rows, G, M, N, K, C=np.full((G, M, N), PRIOR))
    assert np.array_equal(out.cpu().double().numpy(), ref)


@pytest.mark.parametrize("name", sorted(synthetic.GROUPED_WORKLOADS))
def test_grouped_workloads_full_size_sampled(b, name):
    """The grouped workloads at full size, in the bench's launch
    configuration; the oracle computes a seeded sample of cells of every
    group one by one."""
    w = synthetic.GROUPED_WORKLOADS[name]
    A, B = synthetic.grouped_operands(w)
    counts = w.counts()
    dA, dB = A.cuda(), B.cuda()
    out = torch.full((w.groups, w.M, w.N), PRIOR, dtype=torch.float32, device="cuda")
    b.grouped_gemm(dA, dB, counts.cuda(), out=out)
    b.check(b.gemm_get_device_status(0))
    rng = np.random.default_rng(39)
    for g in range(w.groups):
        r = int(counts[g])
        if r == 0:
            continue
        ri = rng.integers(0, r, size=24)
        ci = rng.integers(0, w.N, size=24)
        ref = oracle.gemm_cells(A[g], B[g], r, w.N, w.K, ri, ci)
        got = out[g, torch.as_tensor(ri).cuda(), torch.as_tensor(ci).cuda()].cpu().double().numpy()
        assert np.all(np.abs(got - ref) <= 1e-3 * np.sqrt(w.K)), (g, np.abs(got - ref).max())
        tail = out[g, r:].cpu()
        assert bool((tail == PRIOR).all()), f"group {g}: rows past the count were written"

"""The GEMM entry point that allocates nothing, checked against the ordinary one.

Some callers cannot allocate device memory while they run: allocators or
memory managers that call this library and may not re-enter themselves, and
hosts that reserved all of the GPU's memory up front.  For them
``gemm_f16_f32acc_splitk_noalloc`` keeps its split-K partial sums in a fixed
16 MiB array compiled into the library instead of taking workspace from a
memory pool.  These tests call it through the C ABI twice in a row, with
different inputs so that the second call cannot pass on the first call's
leftover partials, and compare each result with ``gemm_f16_f32acc`` within
the tolerance the other tests use, and -- on small-integer inputs, whose
sums are exact in f32 -- with the oracle bit for bit.  They also check that
a plan needing more than the array holds is refused, and that a call leaves
the device's free memory unchanged.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tiled_staged_matmul_gb300 import synthetic

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.fail("the GPU tests need a CUDA device")
    from tiled_staged_matmul_gb300 import binding
    return binding


def _pad(n, m):
    return -(-n // m) * m


def _both(b, M, N, K, seed, split_k, dist="uniform", with_operands=False):
    """The no-allocation result and the ordinary one, for one seeded input
    (and the CPU operands, with ``with_operands``)."""
    A, B = synthetic.operands(M, N, K, dist, seed=seed)
    lda, ldb, ldc = _pad(K, 8), _pad(N, 8), _pad(N, 4)
    dA = torch.zeros((M, lda), dtype=torch.float16, device="cuda")
    dB = torch.zeros((K, ldb), dtype=torch.float16, device="cuda")
    dA[:, :K] = A.cuda()
    dB[:, :N] = B.cuda()
    c_noalloc = torch.full((M, ldc), float("nan"), dtype=torch.float32, device="cuda")
    c_regular = torch.full((M, ldc), float("nan"), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    b.check(b.gemm_f16_f32acc_splitk_noalloc(dA.data_ptr(), dB.data_ptr(), c_noalloc.data_ptr(),
                                             M, N, K, lda, ldb, ldc, split_k, s))
    opts = b.GemmOptions(split_k, 0, 0, 0)
    b.check(b.gemm_f16_f32acc_opts(dA.data_ptr(), dB.data_ptr(), c_regular.data_ptr(), M, N, K,
                                   lda, ldb, ldc, 0, 0, 0, 1, opts, s))
    b.check(b.gemm_get_device_status(s))
    out = c_noalloc[:, :N].cpu().double().numpy(), c_regular[:, :N].cpu().double().numpy()
    return out + (A, B) if with_operands else out


def _within_tolerance(got, ref, K):
    assert np.all(np.isfinite(got))
    err = float(np.abs(got - ref).max())
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    assert err <= 1e-3 * math.sqrt(K), err
    assert rel <= 1e-4, rel


@pytest.mark.parametrize("M,N,K,split_k", [(256, 256, 65536, 0), (300, 250, 5000, 4)])
def test_two_calls_in_a_row_match_the_ordinary_entry_point(b, M, N, K, split_k):
    plan = b.gemm_plan(M, N, K, 1, b.GemmOptions(split_k, 0, 0, 0))
    assert plan["split_k"] > 1
    # Left to the planner, the no-allocation call lowers the split until the
    # partials fit the scratch; either way it must still split (use the scratch).
    per_split = M * _pad(N, 4) * 4
    used = plan["split_k"] if plan["workspace_bytes"] <= SCRATCH_BYTES else SCRATCH_BYTES // per_split
    assert used > 1 and used * per_split <= SCRATCH_BYTES
    for seed in (101, 202):
        got, ref = _both(b, M, N, K, seed, split_k)
        _within_tolerance(got, ref, K)


@pytest.mark.parametrize("M,N,K,split_k", [(256, 256, 65536, 0), (300, 250, 5000, 4)])
def test_small_integer_splits_exact_against_the_oracle(b, M, N, K, split_k):
    """Split plans on small-integer inputs: both entry points bit for bit
    equal to the oracle, on two calls in a row with different inputs."""
    for seed in (303, 404):
        got, regular, A, B = _both(b, M, N, K, seed, split_k, dist="int4", with_operands=True)
        ref = oracle.gemm_f64(A, B, M, N, K)
        assert np.array_equal(got, ref)
        assert np.array_equal(regular, ref)


def test_plan_larger_than_the_scratch_is_refused(b):
    M = N = 1024
    K = 8192
    dA = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    dB = torch.zeros((K, N), dtype=torch.float16, device="cuda")
    dC = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    st = b.gemm_f16_f32acc_splitk_noalloc(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), M, N, K,
                                          K, N, N, 8, 0)  # 8 x 1024 x 1024 x 4 B = 32 MiB
    assert st == b.GEMM_ERR_INVALID_VALUE
    assert "static scratch" in b.gemm_last_error_string()


def test_call_leaves_free_device_memory_unchanged(b):
    M, N, K = 256, 256, 65536
    A, B = synthetic.operands(M, N, K, "uniform", seed=7)
    dA, dB = A.cuda(), B.cuda()
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    args = (dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), M, N, K, K, N, N, 0, s)
    b.check(b.gemm_f16_f32acc_splitk_noalloc(*args))  # first call on the device: set-up
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        b.check(b.gemm_f16_f32acc_splitk_noalloc(*args))
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    b.check(b.gemm_get_device_status(s))
    assert free_after == free_before


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 1024), (2304, 2304, 320)])
def test_column_slice_tail_without_split(b, M, N, K):
    """Shapes whose no-allocation plan keeps whole K (no partials to hold) but
    cuts the last wave's tiles into column slices: exact on small integers,
    and no scratch involved."""
    plan = b.gemm_plan(M, N, K, 1, b.GemmOptions(0, 0, 0, 0, 0, 1))
    assert plan["split_k"] == 1 and plan["tail_narrow"] == 1 and plan["workspace_bytes"] == 0, plan
    A, B = synthetic.operands(M, N, K, "int4", seed=M + K)
    dA, dB = A.cuda().contiguous(), B.cuda().contiguous()
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    b.check(b.gemm_f16_f32acc_splitk_noalloc(dA.data_ptr(), dB.data_ptr(), C.data_ptr(),
                                             M, N, K, K, N, N, 0, s))
    b.check(b.gemm_get_device_status(s))
    ref = oracle.gemm_f64(A, B, M, N, K)
    assert np.array_equal(C.cpu().double().numpy(), ref)

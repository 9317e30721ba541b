"""The split-K sum taken in thread-block clusters, on a GB300.

Clusters of 2 or 4 CTAs hold consecutive K ranges of one 128-row tile and
add their partials through distributed shared memory before one partial per
cluster goes through the workspace ("A Dumb Triton Runtime Error", section
"The Takeaway and the Final Fix": the inter-CTA reduction is where the cost
sits; the sum stays in a fixed order, never atomics onto C).  The order is
fixed -- a cluster's ranges in ascending order, then the clusters in
ascending order -- so small-integer inputs (exact in f32) must match the
oracle bit for bit for every cluster size, split and tile width, and a
given plan must give bitwise the same C on every run.  Random inputs are
held to the GEMM tolerance."""
import numpy as np
import pytest
import torch

import oracle
from tiled_staged_matmul_gb300 import synthetic
from tiled_staged_matmul_gb300.synthetic import WORKLOADS, integer_twin

from gpu_util import check_exact, check_tolerance, run_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.fail("the GPU tests need a CUDA device")
    from tiled_staged_matmul_gb300 import binding
    return binding


def ref_of(A, B):
    M, K = A.shape
    return oracle.gemm_f64(A.contiguous(), B.contiguous(), M, B.shape[1], K)


def plan_of(b, M, N, K, cl, split_k=0, tile_n=128):
    o = b.GemmOptions(split_k, tile_n, 0, 0, 128)
    o.red_cluster = cl
    return b.gemm_plan(M, N, K, 1, o)


@pytest.mark.parametrize("cl,tile_n", [(2, 128), (4, 128), (4, 256)])
def test_long_K_workload_integer_exact(b, cl, tile_n):
    w = integer_twin(WORKLOADS["gemm_256x256x65536_uniform"])
    p = plan_of(b, w.M, w.N, w.K, cl, tile_n=tile_n)
    assert p["red_cluster"] == cl and p["split_k"] // cl > 1, p
    A, B = synthetic.workload_operands(w)
    C, dC = run_gemm(b, A, B, tile_m=128, tile_n=tile_n, red_cluster=cl)
    check_exact(C.numpy(), ref_of(A, B))
    assert dC.outside_untouched()


@pytest.mark.parametrize("M,N,K,cl,split_k,tile_n", [
    (256, 256, 16384, 4, 8, 128),     # two clusters per tile
    (256, 256, 16384, 2, 16, 128),    # eight pairs per tile
    (128, 128, 1024, 4, 4, 128),      # one cluster holds the whole K: writes C itself
    (128, 128, 1024, 2, 2, 256),      # the same with a pair, a 256-wide tile cut at N
    (200, 300, 20000, 4, 12, 128),    # ragged M and N: rows and columns past the edge
    (70, 77, 9000, 4, 20, 128),       # M below the owned rows of two ranks, N % 4 != 0
    (300, 250, 30000, 2, 16, 256),    # eight pairs per tile over 3 x 1 tiles
    (513, 129, 8192, 4, 8, 128),      # one row and one column past a tile edge
])
def test_integer_exact_across_shapes(b, M, N, K, cl, split_k, tile_n):
    p = plan_of(b, M, N, K, cl, split_k, tile_n)
    assert (p["red_cluster"], p["split_k"]) == (cl, split_k), p
    A, B = synthetic.operands(M, N, K, "int4", seed=M * 7 + N)
    C, dC = run_gemm(b, A, B, split_k=split_k, tile_m=128, tile_n=tile_n, red_cluster=cl)
    check_exact(C.numpy(), ref_of(A, B))
    assert dC.outside_untouched()


@pytest.mark.parametrize("cl", [2, 4])
def test_long_K_workload_random_reproducible(b, cl):
    w = WORKLOADS["gemm_256x256x65536_uniform"]
    A, B = synthetic.workload_operands(w)
    C1, dC = run_gemm(b, A, B, tile_m=128, tile_n=128, red_cluster=cl)
    check_tolerance(C1.numpy(), ref_of(A, B), w.K)
    assert dC.outside_untouched()
    for _ in range(3):
        C2, _ = run_gemm(b, A, B, tile_m=128, tile_n=128, red_cluster=cl)
        assert torch.equal(C1, C2), "the cluster sum is not reproducible run to run"


@pytest.mark.parametrize("act,out", [("gelu", "bf16"), ("relu", "f32"), ("silu", "f16")])
def test_fused_epilogue_through_the_cluster_sum(b, act, out):
    """act(alpha * A.B + bias) applied once to the cluster-summed value."""
    from test_epilogue_gpu import check_epilogue, run_fused
    M, N, K = 256, 200, 30000
    A, B = synthetic.operands(M, N, K, "uniform", seed=77)
    bias = torch.linspace(-0.5, 0.5, N, dtype=torch.float32)
    o = b.GemmOptions(0, 128, 0, 0, 128)
    o.red_cluster = 4
    p = b.gemm_plan(M, N, K, 1, o)
    assert p["red_cluster"] == 4, p
    C, pad_ok = run_fused(b, A, B, ldc_pad=8, alpha=0.5, bias=bias, act=act, out=out, opts=o)
    check_epilogue(C, ref_of(A, B), 0.5, bias.double().numpy(), act, out, K)
    assert pad_ok


def test_stalled_cluster_sum_times_out_and_the_next_call_is_exact(b):
    M, N, K = 256, 256, 8192
    A, B = synthetic.operands(M, N, K, "int4", seed=33)
    dA, dB = A.cuda(), B.cuda()
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream

    def opts(stall, timeout_ms):
        o = b.GemmOptions(8, 128, timeout_ms, stall, 128)
        o.red_cluster = 4
        return o
    assert b.gemm_plan(M, N, K, 1, opts(0, 0))["red_cluster"] == 4
    assert b.gemm_get_device_status(s) == b.GEMM_OK
    assert b.gemm_f16_f32acc_opts(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), M, N, K, K, N, N,
                                  0, 0, 0, 1, opts(1, 200), s) == b.GEMM_OK
    assert b.gemm_get_device_status(s) == b.GEMM_ERR_DEVICE_TIMEOUT
    assert "epilogue" in b.gemm_last_error_string()
    assert b.gemm_get_device_status(s) == b.GEMM_OK
    b.check(b.gemm_f16_f32acc_opts(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), M, N, K, K, N, N,
                                   0, 0, 0, 1, opts(0, 0), s))
    b.check(b.gemm_get_device_status(s))
    assert np.array_equal(dC.cpu().numpy().astype(np.float64), oracle.gemm_f64(A, B, M, N, K))

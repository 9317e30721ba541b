"""Failure detection on the GPU without a GPU fault.

The test hook ``inject_stall`` makes the epilogue wait on a barrier that
nothing ever signals.  The kernel's bounded wait must run out after the
requested limit, record GEMM_ERR_DEVICE_TIMEOUT in the device status word,
wind down (its loads, MMAs and stores drained, TMEM freed) and return; the
context stays usable and the next call is exact again."""
import time

import numpy as np
import pytest
import torch

import oracle
from tiled_staged_matmul_gb300 import synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.fail("the GPU tests need a CUDA device")
    from tiled_staged_matmul_gb300 import binding
    return binding


@pytest.mark.parametrize("M,N,K,split_k,tile_m,tile_n", [
    (512, 512, 1024, 1, 0, 0),        # one CTA per tile
    (256, 256, 8192, 4, 0, 0),        # split K, one CTA per tile
    (512, 512, 1024, 1, 256, 256),    # CTA pairs
    (256, 256, 8192, 4, 256, 256),    # CTA pairs, split-K summed in the kernel
    (256, 256, 8192, 8, 128, 128),    # one CTA per tile, split-K summed in the kernel
    (2304, 2304, 1024, 0, 256, 256),  # CTA pairs with a split tail (opt-in)
])
def test_stalled_wait_times_out_and_the_next_call_is_exact(b, M, N, K, split_k, tile_m, tile_n):
    A, B = synthetic.operands(M, N, K, "int4", seed=31)
    dA, dB = A.cuda(), B.cuda()
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert b.gemm_get_device_status(s) == b.GEMM_OK
    t0 = time.time()
    st = b.gemm_f16_f32acc_opts(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), M, N, K, K, N, N,
                                0, 0, 0, 1, b.GemmOptions(split_k, tile_n, 200, 1, tile_m, 0, 0, 1), s)
    assert st == b.GEMM_OK  # queued; the failure shows on the device
    st = b.gemm_get_device_status(s)
    elapsed = time.time() - t0
    assert st == b.GEMM_ERR_DEVICE_TIMEOUT, b.gemm_status_string(st)
    assert "epilogue" in b.gemm_last_error_string()
    assert elapsed < 20.0
    # the status word was cleared, and the context is healthy
    assert b.gemm_get_device_status(s) == b.GEMM_OK
    st = b.gemm_f16_f32acc_opts(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), M, N, K, K, N, N,
                                0, 0, 0, 1, b.GemmOptions(split_k, tile_n, 0, 0, tile_m, 0, 0, 1), s)
    b.check(st)
    b.check(b.gemm_get_device_status(s))
    ref = oracle.gemm_f64(A, B, M, N, K)
    assert np.array_equal(dC.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("tile_m,tile_n", [(128, 128), (256, 256)])
def test_stalled_grouped_call_times_out_and_the_next_call_is_exact(b, tile_m, tile_n):
    G, M, N, K = 4, 300, 256, 512
    rows = [300, 0, 129, 17]
    A, B = synthetic.operands(M, N, K, "int4", seed=41, batch=G)
    dA, dB = A.cuda(), B.cuda()
    dC = torch.zeros((G, M, N), dtype=torch.float32, device="cuda")
    counts = torch.tensor(rows, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream

    def call(stall, timeout_ms):
        return b.gemm_f16_f32acc_grouped_opts(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(),
                                              counts.data_ptr(), G, M, N, K, K, N, N, M * K, K * N,
                                              M * N, b.GemmOptions(0, tile_n, timeout_ms, stall,
                                                                   tile_m), s)
    assert b.gemm_get_device_status(s) == b.GEMM_OK
    assert call(1, 200) == b.GEMM_OK
    assert b.gemm_get_device_status(s) == b.GEMM_ERR_DEVICE_TIMEOUT
    assert b.gemm_get_device_status(s) == b.GEMM_OK
    b.check(call(0, 0))
    b.check(b.gemm_get_device_status(s))
    ref = oracle.grouped_gemm_f64(A, B, rows, G, M, N, K, C=np.zeros((G, M, N)))
    assert np.array_equal(dC.cpu().numpy().astype(np.float64), ref)

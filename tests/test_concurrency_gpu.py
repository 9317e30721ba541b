"""Concurrent and captured calls on the GPU.

The in-kernel split-K sum keeps its arrival counters in the call's own pool
workspace and zeroes them inside the kernel under a per-launch epoch, so
calls that run at the same time on different streams, and calls replayed
from a CUDA graph, must each get exactly their own sums.  Small-integer
inputs make every result exact, so any cross-talk shows as a wrong cell."""
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


def test_fused_split_K_calls_on_four_streams_at_once(b):
    M, N, K = 256, 256, 32768
    plan = b.gemm_plan(M, N, K, 1, None)
    assert plan["split_k"] > 1 and plan["fused_reduce"]
    problems = [synthetic.operands(M, N, K, "int4", seed=900 + i) for i in range(4)]
    dev = [(A.cuda(), B.cuda(), torch.empty((M, N), dtype=torch.float32, device="cuda"))
           for A, B in problems]
    streams = [torch.cuda.Stream() for _ in problems]
    torch.cuda.synchronize()
    for rep in range(3):
        for (dA, dB, dC), s in zip(dev, streams):
            dC.fill_(float("nan"))
        torch.cuda.synchronize()
        for (dA, dB, dC), s in zip(dev, streams):
            b.check(b.gemm_f16_f32acc(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), M, N, K, K, N, N,
                                      s.cuda_stream))
        torch.cuda.synchronize()
        for (A, B), (_, _, dC) in zip(problems, dev):
            ref = oracle.gemm_f64(A, B, M, N, K)
            assert np.array_equal(dC.cpu().numpy().astype(np.float64), ref), f"pass {rep}"
    b.check(b.gemm_get_device_status(0))


def test_captured_in_a_graph_and_replayed(b):
    M, N, K = 256, 256, 32768
    A1, B1 = synthetic.operands(M, N, K, "int4", seed=950)
    A2, B2 = synthetic.operands(M, N, K, "int4", seed=951)
    dA = A1.cuda()
    dB = B1.cuda()
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        # first call on this stream outside the capture (device state, kernel attributes)
        b.check(b.gemm_f16_f32acc(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), M, N, K, K, N, N,
                                  s.cuda_stream))
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        b.check(b.gemm_f16_f32acc(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), M, N, K, K, N, N,
                                  s.cuda_stream))
    for A, B in ((A1, B1), (A2, B2), (A1, B1)):
        dA.copy_(A)
        dB.copy_(B)
        dC.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(dC.cpu().numpy().astype(np.float64), oracle.gemm_f64(A, B, M, N, K))
    b.check(b.gemm_get_device_status(0))

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU")


# ---------------------------------------------------------------- full-size references
#
# The fp64 oracle over the whole 8192^3 workload costs about 20 s on 16 host
# cores, so it runs once per session and the parity tests that check that
# workload (plain, small-integer twin, fused epilogue, repacked pitches)
# compare every cell against the same reference.

import pytest  # noqa: E402


def _full_reference(name: str, integer: bool):
    import oracle
    from tiled_staged_matmul_gb300 import synthetic
    w = synthetic.WORKLOADS[name]
    if integer:
        w = synthetic.integer_twin(w)
    A, B = synthetic.workload_operands(w)
    return w, A, B, oracle.gemm_f64(A, B, w.M, w.N, w.K)


@pytest.fixture(scope="session")
def full_8192():
    """(workload, A, B, the oracle's C in fp64) of 8192^3, N(0, 1/sqrt(K))."""
    return _full_reference("gemm_8192x8192x8192_normal_invsqrtk", False)


@pytest.fixture(scope="session")
def full_8192_int():
    """The same for the small-integer twin (every cell exact in f32)."""
    return _full_reference("gemm_8192x8192x8192_normal_invsqrtk", True)

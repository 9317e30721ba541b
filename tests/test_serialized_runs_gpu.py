"""The same work with and without serialised launches gives the same bits.

A race between the kernels of one call (a reduction reading a partial that
is not yet written, counters that are not reset in time) can hide while the
GPU runs the work in its usual order and show only when the launches are
serialised, or the other way round ("ADR-1501 ...", section "Context": a
probe raced on an out-of-order queue and only serialising it exposed the
race).  The cases in serial_cases.py -- split-K summed in the kernel, in
clusters, in a second kernel and over a partial last wave, a batched split,
the 256 x 512 tile and a grouped call -- run once in a child process with
CUDA_LAUNCH_BLOCKING=1 and once here without it, and every C must be
bitwise the same."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_serialised_launches_give_bitwise_the_same_results(tmp_path):
    if not torch.cuda.is_available():
        pytest.fail("the GPU tests need a CUDA device")
    sys.path.insert(0, HERE)
    import serial_cases

    out = tmp_path / "serialised.pt"
    env = dict(os.environ, CUDA_LAUNCH_BLOCKING="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "serial_cases.py"), str(out)], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    serial = torch.load(out)
    here = serial_cases.run_all()
    assert set(serial) == set(here)
    for name in here:
        assert torch.equal(serial[name], here[name]), f"{name}: serialised run differs"
        assert torch.isfinite(here[name]).all(), name

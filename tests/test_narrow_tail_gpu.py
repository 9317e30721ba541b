"""Narrow tails on a GB300: plans whose partial last wave is cut into column
slices (halves or quarters of a tile, each over all of K) instead of K
ranges.  Checked against the fp64 oracle: bit for bit on small-integer
inputs, within max |C - C_ref| <= 1e-3 sqrt(K) and relative Frobenius error
<= 1e-4 on random ones, with the fused epilogue, on batches, and where the
last slice of a ragged tile column starts at or past N (nothing stored
there, the accumulator still handed back)."""
import math

import numpy as np
import pytest
import torch

import oracle
from tiled_staged_matmul_gb300 import synthetic

from gpu_util import check_exact, check_tolerance, run_gemm
from test_epilogue_gpu import check_epilogue, run_fused

pytestmark = pytest.mark.gpu

NARROW = 3  # gemm_options_t.split_tail: column slices whenever they apply


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.fail("the GPU tests need a CUDA device")
    from tiled_staged_matmul_gb300 import binding
    return binding


def ref_of(A, B):
    M, K = A.shape
    N = B.shape[1]
    return oracle.gemm_f64(A.contiguous(), B.contiguous(), M, N, K)


def narrow_plan(b, M, N, K, tile_m, tile_n, batch=1):
    opts = b.GemmOptions(0, tile_n, 0, 0, tile_m, 0, 0, NARROW)
    return b.gemm_plan(M, N, K, batch, opts)


# (M, N, K, tile_m, tile_n, pieces): pair tiles cut in halves, one-CTA tiles
# in halves or quarters; the ragged ones have slices that start past N.
CASES = [
    (2304, 2304, 320, 256, 256, 2),    # 81 pair tiles, 5 cut in halves
    (200, 19812, 192, 256, 256, 2),    # one tile row: the last tile's second half starts past N
    (1280, 4096, 256, 128, 256, 4),    # 160 tiles, 8 cut in quarters
    (1280, 3910, 256, 128, 256, 4),    # ... the last tile column 70 wide: two quarters past N
    (1280, 2048, 256, 128, 128, 2),    # 160 tiles of 128 x 128, 8 cut in halves
    (1290, 2030, 200, 128, 128, 2),    # ragged M, N and K
]


@pytest.mark.parametrize("M,N,K,tile_m,tile_n,pieces", CASES)
def test_narrow_tail_integer_bit_exact(b, M, N, K, tile_m, tile_n, pieces):
    plan = narrow_plan(b, M, N, K, tile_m, tile_n)
    assert plan["tail_narrow"] == 1 and plan["tail_split"] == pieces, plan
    assert plan["workspace_bytes"] == 0 and not plan["fused_reduce"]
    A, B = synthetic.operands(M, N, K, "int4", seed=M + N + K)
    C, dC = run_gemm(b, A, B, tile_m=tile_m, tile_n=tile_n, split_tail=NARROW)
    check_exact(C.numpy(), ref_of(A, B))
    assert dC.outside_untouched()


@pytest.mark.parametrize("M,N,K,tile_m,tile_n,pieces", CASES[:4])
def test_narrow_tail_random_within_tolerance(b, M, N, K, tile_m, tile_n, pieces):
    A, B = synthetic.operands(M, N, K, "normal", seed=M + N + K + 1)
    C, dC = run_gemm(b, A, B, tile_m=tile_m, tile_n=tile_n, split_tail=NARROW)
    ref = ref_of(A, B)
    check_tolerance(C.numpy(), ref, K)
    assert dC.outside_untouched()
    # and the same result, within the bound, as whole tiles
    C_whole, _ = run_gemm(b, A, B, tile_m=tile_m, tile_n=tile_n, split_tail=2)
    diff = np.abs(C.numpy().astype(np.float64) - C_whole.numpy())
    assert diff.max() <= 1e-3 * math.sqrt(K)


def test_narrow_tail_batched(b):
    # 2 x 40 pair tiles = 80 on 76 clusters: the last 4 (all in the second
    # matrix) cut in halves; the tile index runs over the whole batch.
    M, N, K, batch = 2048, 1280, 192, 2
    plan = narrow_plan(b, M, N, K, 256, 256, batch)
    assert plan["tail_narrow"] == 1 and plan["tail_tiles"] == 4, plan
    A, B = synthetic.operands(M, N, K, "int4", seed=91, batch=batch)
    C, dC = run_gemm(b, A, B, batch=batch, sA=M * K + 64, sB=K * N + 64, sC=M * N + 20,
                     tile_m=256, tile_n=256, split_tail=NARROW)
    for i in range(batch):
        check_exact(C[i].numpy(), ref_of(A[i], B[i]))
    assert dC.outside_untouched()


# N a multiple of 8 (B and C addressable by the TMA without repacking), the
# ragged ones still with slices past N: 19776 = 77 x 256 + 64, 3912 = 15 x 256 + 72.
@pytest.mark.parametrize("M,N,K,tile_m,tile_n,out", [
    (2304, 2304, 320, 256, 256, "bf16"), (200, 19776, 192, 256, 256, "f16"),
    (1280, 3912, 256, 128, 256, "f32")])
def test_narrow_tail_with_fused_epilogue(b, M, N, K, tile_m, tile_n, out):
    plan = narrow_plan(b, M, N, K, tile_m, tile_n)
    assert plan["tail_narrow"] == 1, plan
    A, B = synthetic.operands(M, N, K, "uniform", seed=M + 5)
    rng = np.random.default_rng(M + 6)
    bias = rng.uniform(-0.5, 0.5, size=N).astype(np.float32)
    opts = b.GemmOptions(0, tile_n, 0, 0, tile_m, 0, 0, NARROW)
    C, pad_ok = run_fused(b, A, B, ldc_pad=8, alpha=0.5, bias=bias, act="gelu", out=out, opts=opts)
    acc = oracle.gemm_f64(A, B, M, N, K)
    check_epilogue(C, acc, 0.5, bias.astype(np.float64), "gelu", out, K)
    assert pad_ok


@pytest.mark.parametrize("M,N,K,batch", [(4096, 4096, 1024, 1), (2304, 2304, 320, 1), (1536, 2048, 1024, 2)])
def test_planner_default_column_slices(b, M, N, K, batch):
    """Shapes whose default plan (no options) cuts the last wave into column
    slices: pair tiles in halves, one-CTA tiles in quarters, a batch."""
    plan = b.gemm_plan(M, N, K, batch)
    assert plan["tail_narrow"] == 1, plan
    A, B = synthetic.operands(M, N, K, "int4", seed=M + 2 * N + K, batch=batch)
    if batch == 1:
        C, dC = run_gemm(b, A, B)
        check_exact(C.numpy(), ref_of(A, B))
    else:
        C, dC = run_gemm(b, A, B, batch=batch, sA=M * K + 64, sB=K * N + 64, sC=M * N + 20)
        for i in range(batch):
            check_exact(C[i].numpy(), ref_of(A[i], B[i]))
    assert dC.outside_untouched()


@pytest.mark.parametrize("tile_m,tile_n,pieces", [(256, 256, 2), (0, 0, 4)])
def test_narrow_tail_batched_with_a_bias_per_batch(b, tile_m, tile_n, pieces):
    """A batch of two whose last wave's tiles (all in the second matrix) are
    cut into column slices, with a bias per batch and GELU into bf16: each
    slice takes the bias row of its own batch."""
    M, N, K, batch = 2048, 1280, 192, 2
    opts = b.GemmOptions(0, tile_n, 0, 0, tile_m, 0, 0, NARROW)
    plan = b.gemm_plan(M, N, K, batch, opts)
    assert plan["tail_narrow"] == 1 and plan["tail_split"] == pieces, plan
    A, B = synthetic.operands(M, N, K, "uniform", seed=93, batch=batch)
    bias = np.random.default_rng(94).uniform(-1, 1, size=(batch, N)).astype(np.float32)
    C, pad_ok = run_fused(b, A, B, alpha=0.5, bias=bias, act="gelu", out="bf16", batch=batch,
                          opts=opts)
    acc = np.stack([oracle.gemm_f64(A[i], B[i], M, N, K) for i in range(batch)])
    check_epilogue(C, acc, 0.5, bias.astype(np.float64), "gelu", "bf16", K)
    assert pad_ok


def test_narrow_tail_through_repacked_operands(b):
    """Odd row pitches (A and B not addressable by the TMA): the operands are
    repacked and the repacked call plans its own column-slice tail."""
    M, N, K = 2304, 2304, 320
    plan = b.gemm_plan(M, N, K, 1)
    assert plan["tail_narrow"] == 1, plan
    A, B = synthetic.operands(M, N, K, "int4", seed=97)
    C, dC = run_gemm(b, A, B, lda=K + 1, ldb=N + 3, ldc=N + 1)
    check_exact(C.numpy(), ref_of(A, B))
    assert dC.outside_untouched()

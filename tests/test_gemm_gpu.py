"""Parity of the CUDA path with the oracle, on a GB300.

Every case runs through the C ABI on padded device buffers (NaN in every
operand's padding and guard band, a sentinel around C) and compares with
the fp64 oracle: bit for bit on small-integer inputs (exact in f32), within
max |C - C_ref| <= 1e-3 sqrt(K) and relative Frobenius error <= 1e-4 on
random inputs.  The shapes span several tiles and ragged tails; the five
workload shapes run at full size, every cell checked."""
import math

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


# (tile_m, tile_n): one CTA per 128-row tile, or a CTA pair per 256-row tile
# (256 x 512: the pair's single-accumulator tile, two MMAs per k-step)
TILES = [(128, 64), (128, 128), (128, 256), (256, 128), (256, 256), (256, 512)]


def ref_of(A, B):
    M, K = A.shape
    N = B.shape[1]
    return oracle.gemm_f64(A.contiguous(), B.contiguous(), M, N, K)


# ---------------------------------------------------------------- the workload shapes

def test_small_shape_integer_bit_exact(b):
    w = WORKLOADS["gemm_64x128x128_int4"]
    A, B = synthetic.workload_operands(w)
    C, dC = run_gemm(b, A, B)
    check_exact(C.numpy(), ref_of(A, B))
    assert dC.outside_untouched()


def test_small_shape_uniform(b):
    w = WORKLOADS["gemm_64x128x128_uniform"]
    A, B = synthetic.workload_operands(w)
    C, dC = run_gemm(b, A, B)
    check_tolerance(C.numpy(), ref_of(A, B), w.K)
    assert dC.outside_untouched()


def test_1000_cube_ragged_edges(b):
    w = WORKLOADS["gemm_1000x1000x1000_normal"]
    A, B = synthetic.workload_operands(w)
    C, dC = run_gemm(b, A, B)
    check_tolerance(C.numpy(), ref_of(A, B), w.K)
    assert dC.outside_untouched()


def test_1000_cube_integer_bit_exact(b):
    w = integer_twin(WORKLOADS["gemm_1000x1000x1000_normal"])
    A, B = synthetic.workload_operands(w)
    C, _ = run_gemm(b, A, B)
    check_exact(C.numpy(), ref_of(A, B))


def test_4096_cube(b):
    w = WORKLOADS["gemm_4096x4096x4096_normal_invsqrtk"]
    A, B = synthetic.workload_operands(w)
    C, dC = run_gemm(b, A, B)
    check_tolerance(C.numpy(), ref_of(A, B), w.K)
    assert dC.outside_untouched()


def test_4096_cube_integer_bit_exact(b):
    """The integer twin at full size in the default plan (the last wave's
    tiles split along K and summed in the kernel): exact in f32."""
    w = integer_twin(WORKLOADS["gemm_4096x4096x4096_normal_invsqrtk"])
    assert b.gemm_plan(w.M, w.N, w.K)["tail_split"] >= 2
    A, B = synthetic.workload_operands(w)
    C, dC = run_gemm(b, A, B)
    check_exact(C.numpy(), ref_of(A, B))
    assert dC.outside_untouched()


def test_long_K_split(b):
    w = WORKLOADS["gemm_256x256x65536_uniform"]
    plan = b.gemm_plan(w.M, w.N, w.K)
    assert plan["split_k"] > 1
    A, B = synthetic.workload_operands(w)
    C, dC = run_gemm(b, A, B)
    check_tolerance(C.numpy(), ref_of(A, B), w.K)
    assert dC.outside_untouched()
    C2, _ = run_gemm(b, A, B)
    assert torch.equal(C, C2), "split-K result is not reproducible run to run"


def test_long_K_integer_bit_exact_for_every_split(b):
    w = integer_twin(WORKLOADS["gemm_256x256x65536_uniform"])
    A, B = synthetic.workload_operands(w)
    ref = ref_of(A, B)
    for tile_m, tile_n in ((128, 128), (256, 256)):
        for s in (1, 2, 3, 7, 64, 0):
            C, _ = run_gemm(b, A, B, split_k=s, tile_m=tile_m, tile_n=tile_n)
            check_exact(C.numpy(), ref)


@pytest.mark.parametrize("M,N,K,tile_m,tile_n,split_k", [
    (256, 256, 65536, 256, 256, 0), (256, 256, 65536, 128, 128, 38), (300, 250, 20000, 256, 128, 0),
    (130, 70, 9000, 128, 64, 11), (1000, 1000, 1000, 256, 128, 2)])
def test_in_kernel_and_separate_reduce_agree_bitwise(b, M, N, K, tile_m, tile_n, split_k):
    """Both reductions sum the splits in ascending order, so they agree bit for bit."""
    plan = b.gemm_plan(M, N, K, 1, b.GemmOptions(split_k, tile_n, 0, 0, tile_m, 0))
    assert plan["split_k"] > 1 and plan["fused_reduce"]
    A, B = synthetic.operands(M, N, K, "uniform", seed=M + K)
    C_in, dC = run_gemm(b, A, B, split_k=split_k, tile_m=tile_m, tile_n=tile_n, splitk_reduce=2)
    C_sep, _ = run_gemm(b, A, B, split_k=split_k, tile_m=tile_m, tile_n=tile_n, splitk_reduce=1)
    assert torch.equal(C_in, C_sep)
    assert dC.outside_untouched()
    check_tolerance(C_in.numpy(), ref_of(A, B), K)


@pytest.mark.parametrize("M,N,K", [(2304, 2304, 1024), (4096, 4096, 1024), (2560, 4096, 1536), (2200, 2270, 832)])
def test_split_tail(b, M, N, K):
    """Plans whose partial last wave is split across all slots: exact on
    integers, and the same within tolerance as whole tiles on random inputs."""
    plan = b.gemm_plan(M, N, K, 1, b.GemmOptions(0, 0, 0, 0, 0, 0, 0, 1))
    assert plan["tail_split"] >= 2, plan
    A, B = synthetic.operands(M, N, K, "int4", seed=M + N)
    C, dC = run_gemm(b, A, B, split_tail=1)
    check_exact(C.numpy(), ref_of(A, B))
    assert dC.outside_untouched()
    A, B = synthetic.operands(M, N, K, "normal", seed=M + N + 1)
    C_tail, _ = run_gemm(b, A, B, split_tail=1)
    C_whole, _ = run_gemm(b, A, B)
    check_tolerance(C_tail.numpy(), ref_of(A, B), K)
    diff = np.abs(C_tail.numpy().astype(np.float64) - C_whole.numpy())
    assert diff.max() <= 1e-3 * math.sqrt(K)


def test_in_kernel_reduce_batched(b):
    M, N, K, batch = 200, 136, 12000, 3
    A, B = synthetic.operands(M, N, K, "int4", seed=23, batch=batch)
    plan = b.gemm_plan(M, N, K, batch)
    assert plan["split_k"] > 1 and plan["fused_reduce"]
    C, dC = run_gemm(b, A, B, batch=batch, sA=M * K + 64, sB=K * 136 + 64, sC=M * 136 + 20)
    for i in range(batch):
        check_exact(C[i].numpy(), ref_of(A[i], B[i]))
    assert dC.outside_untouched()


@pytest.mark.parametrize("tile_m,tile_n", TILES)
def test_every_tile_shape_on_random_inputs(b, tile_m, tile_n):
    A, B = synthetic.operands(700, 900, 1500, "normal", seed=tile_m + tile_n)
    C, dC = run_gemm(b, A, B, tile_m=tile_m, tile_n=tile_n)
    check_tolerance(C.numpy(), ref_of(A, B), 1500)
    assert dC.outside_untouched()


def test_pair_tiles_with_many_units_per_cluster(b):
    # 2048 x 2048 on 256 x 128 pair tiles: 128 units over at most 76 clusters,
    # so clusters walk several tiles and both TMEM accumulators take turns.
    A, B = synthetic.operands(2048, 2048, 512, "int4", seed=17)
    C, _ = run_gemm(b, A, B, tile_m=256, tile_n=128)
    check_exact(C.numpy(), ref_of(A, B))


def test_wide_pair_tile_walks_many_tiles(b):
    # 4096 x 4096 on 256 x 512 tiles: 128 units over at most 76 clusters, so
    # the single accumulator is drained and refilled tile after tile.
    A, B = synthetic.operands(4096, 4096, 512, "int4", seed=29)
    C, dC = run_gemm(b, A, B, tile_m=256, tile_n=512)
    check_exact(C.numpy(), ref_of(A, B))
    assert dC.outside_untouched()


def test_wide_pair_tile_batched(b):
    batch, M, N, K = 3, 600, 1100, 300
    A, B = synthetic.operands(M, N, K, "int4", seed=31, batch=batch)
    C, dC = run_gemm(b, A, B, batch=batch, tile_m=256, tile_n=512)
    for i in range(batch):
        check_exact(C[i].numpy(), ref_of(A[i], B[i]))
    assert dC.outside_untouched()


@pytest.mark.parametrize("M,N,K", [(1536, 2560, 4096), (1000, 1300, 777)])
def test_wide_pair_tile_matches_the_256_wide_tile_bitwise(b, M, N, K):
    # Each output element takes the same MMAs in the same k order in a
    # 256 x 256 and a 256 x 512 tile (whole tiles, no K split), so the two
    # plans agree bit for bit on random inputs.
    A, B = synthetic.operands(M, N, K, "normal", seed=M + 3 * N + K)
    C256, _ = run_gemm(b, A, B, tile_m=256, tile_n=256, split_k=1)
    C512, dC = run_gemm(b, A, B, tile_m=256, tile_n=512, split_k=1)
    assert torch.equal(C256, C512)
    check_tolerance(C512.numpy(), ref_of(A, B), K)
    assert dC.outside_untouched()


def test_8192_cube_every_cell(b, full_8192):
    """The headline workload at full size in its default plan, every cell
    against the fp64 oracle."""
    w, A, B, ref = full_8192
    C, dC = run_gemm(b, A, B)
    check_tolerance(C.numpy(), ref, w.K)
    assert dC.outside_untouched()


def test_8192_cube_wide_pair_tile_every_cell(b, full_8192):
    """The headline workload on the opt-in 256 x 512 pair tile, every cell
    against the fp64 oracle."""
    w, A, B, ref = full_8192
    C, dC = run_gemm(b, A, B, tile_m=256, tile_n=512)
    check_tolerance(C.numpy(), ref, w.K)
    assert dC.outside_untouched()


def test_8192_cube_integer_every_cell_and_transpose_identity(b, full_8192_int):
    """Its small-integer twin: every cell bit for bit against the oracle, and
    (A.B)^T == B^T.A^T exactly by a second call with swapped operands."""
    w, A, B, ref = full_8192_int
    C, _ = run_gemm(b, A, B)
    check_exact(C.numpy(), ref)
    Ct, _ = run_gemm(b, B.t().contiguous(), A.t().contiguous())
    assert torch.equal(C, Ct.t())


# ---------------------------------------------------------------- ragged and edge cases

RAGGED = [(1, 1, 1), (1, 8, 1), (7, 9, 63), (129, 257, 65), (130, 250, 1000),
          (255, 129, 127), (128, 256, 64), (300, 1, 200), (1, 300, 200), (513, 77, 33)]


@pytest.mark.parametrize("M,N,K", RAGGED)
@pytest.mark.parametrize("tile_m,tile_n", TILES)
def test_ragged_integer_bit_exact(b, M, N, K, tile_m, tile_n):
    A, B = synthetic.operands(M, N, K, "int4", seed=M * 7 + N * 13 + K)
    C, dC = run_gemm(b, A, B, tile_n=tile_n, tile_m=tile_m)
    check_exact(C.numpy(), ref_of(A, B))
    assert dC.outside_untouched()


@pytest.mark.parametrize("M,N,K", RAGGED)
def test_ragged_random(b, M, N, K):
    A, B = synthetic.operands(M, N, K, "normal", seed=M + N + K)
    C, dC = run_gemm(b, A, B)
    check_tolerance(C.numpy(), ref_of(A, B), K)
    assert dC.outside_untouched()


@pytest.mark.parametrize("pad", [(8, 0, 0), (0, 16, 4), (24, 8, 12)])
def test_padded_leading_dimensions(b, pad):
    M, N, K = 200, 136, 300
    A, B = synthetic.operands(M, N, K, "int4", seed=5)
    C, dC = run_gemm(b, A, B, lda=304 + pad[0], ldb=136 + pad[1], ldc=136 + pad[2])
    check_exact(C.numpy(), ref_of(A, B))
    assert dC.outside_untouched()


def test_K_zero_writes_zeros(b):
    M, N = 70, 90
    A = torch.zeros((M, 0), dtype=torch.float16)
    B = torch.zeros((0, N), dtype=torch.float16)
    C, dC = run_gemm(b, A, B)
    assert torch.equal(C, torch.zeros(M, N))
    assert dC.outside_untouched()


def test_identity_copies_B(b):
    K, N = 256, 200
    _, B = synthetic.operands(K, N, K, "normal", seed=77)
    A = torch.eye(K, dtype=torch.float16)
    C, _ = run_gemm(b, A, B)
    assert torch.equal(C, B.float())


def test_row_sum_special_case(b):
    """N = 1 with B = ones: the pages' tiled row sum as a GEMM."""
    M, K = 333, 1000
    A, _ = synthetic.operands(M, 1, K, "uniform", seed=3)
    B = torch.ones((K, 1), dtype=torch.float16)
    C, _ = run_gemm(b, A, B)
    check_tolerance(C.numpy(), ref_of(A, B), K)
    x = torch.tensor([[1.0, 1.0, 1.0], [1.0, 1.0, 1.0]], dtype=torch.float16)
    C, _ = run_gemm(b, x, torch.ones((3, 1), dtype=torch.float16))
    assert C[:, 0].tolist() == [3.0, 3.0]


def test_all_ones_give_K(b):
    for (M, N, K) in [(64, 128, 128), (256, 256, 65536)]:
        A = torch.ones((M, K), dtype=torch.float16)
        B = torch.ones((K, N), dtype=torch.float16)
        C, _ = run_gemm(b, A, B)
        assert bool((C == K).all()), (M, N, K)


def test_subnormal_inputs_are_not_flushed(b):
    M = K = 128
    N = 64
    rng = np.random.default_rng(1)
    bits = rng.integers(1, 1024, size=(M, K)).astype(np.uint16)
    A = torch.from_numpy(bits.view(np.float16).copy())
    B = torch.zeros((K, N), dtype=torch.float16)
    B[:N, :N] = torch.eye(N, dtype=torch.float16)
    C, _ = run_gemm(b, A, B)
    assert torch.equal(C, A[:, :N].float())


def test_nan_and_inf_propagate_as_ieee(b):
    """One NaN row and one +Inf entry in A: the CUDA path makes the same cells
    NaN, +Inf and -Inf as the oracle (IEEE: Inf x 0 = NaN, one infinite term
    per cell so the order of the sum does not matter) and the rest exact."""
    from test_oracle_pins import special_values_case
    A, B, nan_cells, pos_inf, neg_inf = special_values_case()
    M, K = A.shape
    N = B.shape[1]
    C, dC = run_gemm(b, torch.from_numpy(A), torch.from_numpy(B))
    C = C.numpy().astype(np.float64)
    ref = oracle.gemm_f64(A, B, M, N, K)
    assert np.array_equal(np.isnan(C), nan_cells)
    assert np.array_equal(np.isposinf(C), pos_inf)
    assert np.array_equal(np.isneginf(C), neg_inf)
    finite = ~(nan_cells | pos_inf | neg_inf)
    assert np.array_equal(C[finite], ref[finite])
    assert dC.outside_untouched()


def test_batched(b):
    for (M, N, K) in [(64, 128, 128), (1000, 1000, 1000)]:
        batch = 3
        A, B = synthetic.operands(M, N, K, "int4", seed=11, batch=batch)
        lda, ldb, ldc = -(-K // 8) * 8, -(-N // 8) * 8, -(-N // 4) * 4
        # gaps between batches (strides larger than one matrix)
        C, dC = run_gemm(b, A, B, batch=batch, lda=lda, ldb=ldb, ldc=ldc,
                         sA=M * lda + 64, sB=K * ldb + 128, sC=M * ldc + 36)
        for i in range(batch):
            check_exact(C[i].numpy(), ref_of(A[i], B[i]))
        assert dC.outside_untouched()


@pytest.mark.parametrize("tile_m", [128, 256])
def test_batched_random_with_split(b, tile_m):
    M, N, K, batch = 256, 192, 8192, 2
    A, B = synthetic.operands(M, N, K, "uniform", seed=12, batch=batch)
    C, _ = run_gemm(b, A, B, batch=batch, split_k=5, tile_m=tile_m, tile_n=128)
    for i in range(batch):
        check_tolerance(C[i].numpy(), ref_of(A[i], B[i]), K)


def test_results_are_reproducible(b):
    w = WORKLOADS["gemm_1000x1000x1000_normal"]
    A, B = synthetic.workload_operands(w)
    C1, _ = run_gemm(b, A, B)
    C2, _ = run_gemm(b, A, B)
    assert torch.equal(C1, C2)


def test_non_default_stream(b):
    A, B = synthetic.operands(300, 200, 500, "int4", seed=9)
    s = torch.cuda.Stream()
    C, _ = run_gemm(b, A, B, stream=s)
    check_exact(C.numpy(), ref_of(A, B))


def test_torch_convenience_wrapper(b):
    A, B = synthetic.operands(190, 210, 336, "int4", seed=10)
    dA = A.cuda()
    dB = torch.zeros((336, 216), dtype=torch.float16, device="cuda")[:, :210]
    dB.copy_(B)
    out = b.gemm(dA, dB)  # N = 210: out gets a padded pitch, returned as a view
    torch.cuda.synchronize()
    assert out.shape == (190, 210) and out.stride(0) % 4 == 0
    check_exact(out.cpu().numpy(), ref_of(A, B))
    # row pitches of 30 and 14 elements: not TMA-addressable, served by repacking
    A2, B2 = synthetic.operands(8, 14, 30, "int4", seed=11)
    out = b.gemm(A2.cuda(), B2.cuda(), torch.empty((8, 14), dtype=torch.float32, device="cuda"))
    check_exact(out.cpu().numpy(), ref_of(A2, B2))
    with pytest.raises(ValueError):
        b.gemm(dA.t(), dB)  # a non-unit last stride


def test_host_pipeline_results(b):
    """Host-resident problems through the double-buffered pipeline: every
    result matches its own inputs, also once buffer sets are reused."""
    M, N, K = 300, 264, 520
    pipe = b.HostPipeline(M, N, K, depth=2)
    problems = [synthetic.operands(M, N, K, "int4", seed=400 + i) for i in range(5)]
    outs = [torch.empty((M, N), dtype=torch.float32).pin_memory() for _ in problems]
    for (A, B), C in zip(problems, outs):
        pipe.submit(A.pin_memory(), B.pin_memory(), C)
    pipe.synchronize()
    for (A, B), C in zip(problems, outs):
        check_exact(C.numpy(), ref_of(A, B))


# ---------------------------------------------------------------- device-side argument checks

def test_host_pointer_rejected(b):
    A = torch.zeros((64, 64), dtype=torch.float16)  # pageable host memory
    dB = torch.zeros((64, 64), dtype=torch.float16, device="cuda")
    dC = torch.zeros((64, 64), dtype=torch.float32, device="cuda")
    st = b.gemm_f16_f32acc(A.data_ptr(), dB.data_ptr(), dC.data_ptr(), 64, 64, 64, 64, 64, 64, 0)
    assert st == b.GEMM_ERR_INVALID_VALUE


def test_allocation_too_small_rejected(b):
    """C claims rows past the end of its allocation: rejected before launch.
    A, B and C share one fresh 64 MiB allocation (A and B at its start), so
    the claimed span of C overlaps neither operand and the allocation-range
    check is what fires."""
    torch.cuda.empty_cache()
    buf = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    base = buf.data_ptr()
    A, B = base, base + (1 << 20)
    C = base + (64 << 20) - 64 * 64 * 4  # exactly 64 x 64 f32 fit before the end
    assert b.gemm_f16_f32acc(A, B, C, 64, 64, 64, 64, 64, 64, 0) == b.GEMM_OK
    assert b.gemm_get_device_status(0) == b.GEMM_OK
    st = b.gemm_f16_f32acc(A, B, C, 128, 64, 64, 64, 64, 64, 0)  # 128 rows do not
    assert st == b.GEMM_ERR_INVALID_VALUE, b.gemm_status_string(st)
    del buf

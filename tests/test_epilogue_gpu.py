"""The fused epilogue on the GPU against the epilogue oracle.

C = act(alpha * A.B + bias[j]) rounded to the output type (f32, f16, bf16).
The reference is the fp64 GEMM through ``oracle.epilogue_f64`` and
``oracle.round_to_out``.  Bound per element: the GEMM's tolerance
(1e-3 sqrt(K)) times |alpha| and the activation's largest slope (1.13 for
GELU; 1.1 for SiLU; 1 otherwise), plus one unit in the last place of the
output type at the value (the GPU rounds its f32 value, the oracle its fp64
value, so the two may land on neighbouring representable values).  Small-
integer inputs with exact scales and biases are checked bit for bit."""
import math

import numpy as np
import pytest
import torch

import oracle
from tiled_staged_matmul_gb300 import synthetic

from gpu_util import SENTINEL

pytestmark = pytest.mark.gpu

ACTS = ["none", "relu", "leaky_relu", "gelu", "gelu_tanh", "silu"]
OUTS = ["f32", "f16", "bf16"]
TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
MANT = {"f32": 23, "f16": 10, "bf16": 7}
MIN_ULP = {"f32": 2.0 ** -149, "f16": 2.0 ** -24, "bf16": 2.0 ** -133}
SLOPE_MAX = {"gelu": 1.13, "silu": 1.1}


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.fail("the GPU tests need a CUDA device")
    from tiled_staged_matmul_gb300 import binding
    return binding


def ulp(x, out):
    x = np.maximum(np.abs(x), 1e-300)
    return np.maximum(2.0 ** (np.floor(np.log2(x)) - MANT[out]), MIN_ULP[out])


def as_f64(t):
    return t.float().cpu().double().numpy()


def check_epilogue(C, acc, alpha, bias, act, out, K, slope=0.01):
    pre = oracle.epilogue_f64(acc, alpha, bias, act, slope)
    ref = oracle.round_to_out(pre, out)
    assert np.all(np.isfinite(C)), "non-finite output"
    bound = SLOPE_MAX.get(act, 1.0) * abs(alpha) * 1e-3 * math.sqrt(max(K, 1)) + ulp(np.maximum(np.abs(ref), np.abs(C)), out)
    err = np.abs(C - ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), f"{act}/{out}: err {err[worst]} > bound {bound[worst]} at {worst}"


def run_fused(b, A, B, *, ldc_pad=0, alpha=1.0, bias=None, act="none", out="f32", slope=0.01,
              opts=None, batch=1):
    """A: (batch,) M x K, B: (batch,) K x N (CPU f16).  C in a sentinel-filled
    buffer with `ldc_pad` extra elements per row; returns (C as fp64 numpy,
    the padding untouched)."""
    M, K = A.shape[-2], A.shape[-1]
    N = B.shape[-1]
    dA, dB = A.cuda().contiguous(), B.cuda().contiguous()
    dt = TORCH[out]
    ldc = N + ldc_pad
    Cbuf = torch.full((batch, M, ldc), SENTINEL if out == "f32" else 1000.0, dtype=dt, device="cuda")
    dbias = torch.as_tensor(bias, dtype=torch.float32).cuda().contiguous() if bias is not None else None
    epi = b.epilogue(alpha, dbias.data_ptr() if dbias is not None else 0,
                     N if dbias is not None and dbias.dim() == 2 else 0, act, slope, out)
    s = torch.cuda.current_stream().cuda_stream
    b.check(b.gemm_f16_fused(dA.data_ptr(), dB.data_ptr(), Cbuf.data_ptr(), M, N, K, K, N, ldc,
                             M * K if batch > 1 else 0, K * N if batch > 1 else 0,
                             M * ldc if batch > 1 else 0, batch, epi, opts, s))
    b.check(b.gemm_get_device_status(s))
    pad_ok = bool((Cbuf[..., N:] == (SENTINEL if out == "f32" else 1000.0)).all())
    C = as_f64(Cbuf[..., :N])
    return (C if batch > 1 else C[0]), pad_ok


@pytest.mark.parametrize("out", OUTS)
@pytest.mark.parametrize("act", ACTS)
def test_every_activation_and_output_type(b, act, out):
    M, N, K = 300, 203, 520
    A, B = synthetic.operands(M, N, K, "uniform", seed=71)
    rng = np.random.default_rng(72)
    bias = rng.uniform(-0.5, 0.5, size=N).astype(np.float32)
    C, pad_ok = run_fused(b, A, B, alpha=0.75, bias=bias, act=act, out=out, slope=0.05)
    acc = oracle.gemm_f64(A, B, M, N, K)
    check_epilogue(C, acc, 0.75, bias.astype(np.float64), act, out, K, slope=0.05)
    assert pad_ok


@pytest.mark.parametrize("out,K", [("f32", 256), ("f16", 64), ("bf16", 8)])
@pytest.mark.parametrize("act,slope", [("relu", 0.0), ("leaky_relu", 0.5), ("none", 0.0)])
def test_integer_inputs_are_exact(b, out, K, act, slope):
    M, N = 192, 136
    A, B = synthetic.operands(M, N, K, "int4", seed=73)
    bias = np.arange(N, dtype=np.float32) % 7 - 3
    C, pad_ok = run_fused(b, A, B, alpha=2.0, bias=bias, act=act, out=out, slope=slope)
    acc = oracle.gemm_f64(A, B, M, N, K)
    ref = oracle.round_to_out(oracle.epilogue_f64(acc, 2.0, bias, act, slope), out)
    assert np.array_equal(C, ref)
    assert pad_ok


@pytest.mark.parametrize("splitk_reduce", [0, 1])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_split_K_sums_get_the_epilogue(b, splitk_reduce, out):
    M, N, K = 256, 264, 16384
    A, B = synthetic.operands(M, N, K, "uniform", seed=74)
    bias = np.linspace(-1, 1, N).astype(np.float32)
    opts = b.GemmOptions(8, 0, 0, 0, 0, splitk_reduce)
    plan = b.gemm_plan(M, N, K, 1, opts)
    assert plan["split_k"] == 8 and (splitk_reduce == 0 or not plan["fused_reduce"])
    C, pad_ok = run_fused(b, A, B, alpha=0.5, bias=bias, act="gelu", out=out, opts=opts)
    acc = oracle.gemm_f64(A, B, M, N, K)
    check_epilogue(C, acc, 0.5, bias, "gelu", out, K)
    assert pad_ok


def test_in_kernel_and_separate_split_sums_agree_bitwise(b):
    M, N, K = 256, 256, 8192
    A, B = synthetic.operands(M, N, K, "uniform", seed=75)
    bias = np.linspace(-1, 1, N).astype(np.float32)
    outs = []
    for red in (0, 1):
        C, _ = run_fused(b, A, B, alpha=1.5, bias=bias, act="silu", out="f16",
                         opts=b.GemmOptions(4, 0, 0, 0, 0, red))
        outs.append(C)
    assert np.array_equal(outs[0], outs[1])


def test_K_zero_gives_the_epilogue_of_the_empty_sum(b):
    M, N = 70, 45
    bias = np.linspace(-2, 2, N).astype(np.float32)
    dbias = torch.as_tensor(bias).cuda()
    C = torch.full((M, 48), 5.0, dtype=torch.float16, device="cuda")
    epi = b.epilogue(3.0, dbias.data_ptr(), 0, "gelu", 0.0, "f16")
    b.check(b.gemm_f16_fused(0, 0, C.data_ptr(), M, N, 0, 8, 48, 48, 0, 0, 0, 1, epi, None, 0))
    b.check(b.gemm_get_device_status(0))
    got = as_f64(C[:, :N])
    ref = oracle.round_to_out(oracle.epilogue_f64(np.zeros((M, N)), 3.0, bias, "gelu"), "f16")
    assert np.all(np.abs(got - ref) <= ulp(np.abs(ref), "f16"))
    assert bool((C[:, N:] == 5.0).all())


def test_batched_with_a_bias_per_batch(b):
    batch, M, N, K = 3, 130, 96, 200
    A, B = synthetic.operands(M, N, K, "uniform", seed=76, batch=batch)
    bias = np.random.default_rng(77).uniform(-1, 1, size=(batch, N)).astype(np.float32)
    C, pad_ok = run_fused(b, A, B, alpha=1.0, bias=bias, act="relu", out="bf16", batch=batch)
    acc = np.stack([oracle.gemm_f64(A[i], B[i], M, N, K) for i in range(batch)])
    check_epilogue(C, acc, 1.0, bias.astype(np.float64), "relu", "bf16", K)
    assert pad_ok


@pytest.mark.parametrize("tile_m,tile_n", [(128, 64), (128, 256), (256, 128), (256, 256), (256, 512)])
def test_every_tile_shape_with_16_bit_output(b, tile_m, tile_n):
    M, N, K = 520, 333, 300
    A, B = synthetic.operands(M, N, K, "uniform", seed=78)
    bias = np.linspace(-1, 1, N).astype(np.float32)
    C, pad_ok = run_fused(b, A, B, alpha=1.0, bias=bias, act="gelu_tanh", out="f16", ldc_pad=3,
                          opts=b.GemmOptions(1, tile_n, 0, 0, tile_m))
    check_epilogue(C, oracle.gemm_f64(A, B, M, N, K), 1.0, bias, "gelu_tanh", "f16", K)
    assert pad_ok


@pytest.mark.parametrize("act,out", [("gelu", "bf16"), ("silu", "f32"), ("leaky_relu", "f16")])
def test_wide_pair_tile_epilogue_matches_the_256_wide_tile_bitwise(b, act, out):
    # Whole tiles and no K split on both: the same sums and the same
    # epilogue arithmetic per element, so the same bits.
    M, N, K = 1000, 1304, 776
    A, B = synthetic.operands(M, N, K, "normal", seed=79)
    bias = np.linspace(-1, 1, N).astype(np.float32)
    outs = [run_fused(b, A, B, alpha=0.5, bias=bias, act=act, out=out, slope=0.1,
                      opts=b.GemmOptions(1, tile_n, 0, 0, 256)) for tile_n in (256, 512)]
    assert np.array_equal(outs[0][0], outs[1][0], equal_nan=True)
    assert outs[1][1]
    check_epilogue(outs[1][0], oracle.gemm_f64(A, B, M, N, K), 0.5, bias, act, out, K, slope=0.1)


def test_repacked_16_bit_output(b):
    M, N, K = 200, 101, 96
    A, B = synthetic.operands(M, N, K, "int4", seed=79)
    C, pad_ok = run_fused(b, A, B, act="relu", out="bf16", ldc_pad=2)   # ldc 103: repacked
    ref = oracle.round_to_out(oracle.epilogue_f64(oracle.gemm_f64(A, B, M, N, K), 1.0, None, "relu"), "bf16")
    assert np.array_equal(C, ref)
    assert pad_ok


@pytest.mark.parametrize("tile_m,tile_n", [(0, 0), (256, 512)])
def test_grouped_with_epilogue_keeps_rows_past_the_counts(b, tile_m, tile_n):
    G, M, N, K = 4, 160, 72, 128
    rows = [160, 0, 33, 100]
    A, B = synthetic.operands(M, N, K, "uniform", seed=80, batch=G)
    bias = np.random.default_rng(81).uniform(-1, 1, size=(G, N)).astype(np.float32)
    out = torch.full((G, M, N), 9.0, dtype=torch.bfloat16, device="cuda")
    counts = torch.tensor(rows, dtype=torch.int32, device="cuda")
    b.grouped_gemm(A.cuda(), B.cuda(), counts, out=out, alpha=0.5,
                   bias=torch.as_tensor(bias).cuda(), activation="silu", tile_m=tile_m, tile_n=tile_n)
    C = as_f64(out)
    for g, r in enumerate(rows):
        assert np.all(C[g, r:] == 9.0)
        if r:
            acc = oracle.gemm_f64(A[g, :r].contiguous(), B[g], r, N, K)
            check_epilogue(C[g, :r], acc, 0.5, bias[g].astype(np.float64), "silu", "bf16", K)


def test_torch_wrapper(b):
    A, B = synthetic.operands(64, 80, 96, "uniform", seed=82)
    bias = torch.linspace(-1, 1, 80).cuda()
    out = b.gemm(A.cuda(), B.cuda(), alpha=2.0, bias=bias, activation="gelu", out_dtype=torch.float16)
    assert out.dtype == torch.float16 and out.shape == (64, 80)
    check_epilogue(as_f64(out), oracle.gemm_f64(A, B, 64, 80, 96), 2.0, bias.cpu().double().numpy(),
                   "gelu", "f16", 96)


@pytest.mark.parametrize("act", ["gelu", "gelu_tanh", "silu", "relu", "leaky_relu"])
def test_activation_accuracy_on_its_own(b, act):
    """K = 1 and B = 1: C = act(a) for a grid of f16 values a, against the
    fp64 definition, within 2e-6 x max(1, |a|) (the product is exact here,
    so this bounds the activation's own f32 evaluation)."""
    xs = np.unique(np.concatenate([np.linspace(-12, 12, 3001), np.linspace(-1, 1, 2001),
                                   [0.0, -0.0, 1e-4, -1e-4, 30.0, -30.0, 80.0, -80.0]]).astype(np.float16))
    M = xs.size
    A = torch.from_numpy(xs.reshape(M, 1).copy())
    B = torch.ones((1, 8), dtype=torch.float16)
    C, _ = run_fused(b, A, B, act=act, out="f32", slope=0.125)
    got = C[:, 0]
    want = oracle.activation_f64(xs.astype(np.float64), act, 0.125)
    err = np.abs(got - want)
    bound = 2e-6 * np.maximum(1.0, np.abs(xs.astype(np.float64)))
    worst = int(np.argmax(err - bound))
    assert np.all(err <= bound), (act, float(xs[worst]), float(got[worst]), float(want[worst]))


@pytest.mark.parametrize("name", ["gemm_4096x4096x4096_normal_invsqrtk", "gemm_256x256x65536_uniform",
                                  "gemm_8192x8192x8192_normal_invsqrtk"])
def test_benchmarked_epilogue_full_size(b, name, request):
    """The fused epilogue the bench times (bias + GELU into bf16) at the
    workloads' full sizes and in their default plans, every cell against the
    epilogue oracle applied to the fp64 product."""
    if name == "gemm_8192x8192x8192_normal_invsqrtk":
        w, A, B, acc = request.getfixturevalue("full_8192")
    else:
        w = synthetic.WORKLOADS[name]
        A, B = synthetic.workload_operands(w)
        acc = oracle.gemm_f64(A, B, w.M, w.N, w.K)
    bias = np.linspace(-1, 1, w.N).astype(np.float32)
    C, pad_ok = run_fused(b, A, B, alpha=1.0, bias=bias, act="gelu", out="bf16")
    check_epilogue(C, acc, 1.0, bias.astype(np.float64), "gelu", "bf16", w.K)
    assert pad_ok

"""The oracle for C = A.B with f16 operands (fp64 accumulation).

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only ``tests/``, the smoke
check in ``__graft_entry__`` and the CPU-baseline / reference legs of
``bench.py`` may import this package.  It shares no code with the CUDA
library (``tiled_staged_matmul_gb300``) and neither side imports the other.

Two independent implementations live here:

* ``gemm_f64`` / ``gemm_cells`` -- the C library ``oracle_gemm.c``: the plain
  triple loop, fp64, ascending k (see the header of that file for the passage
  it follows).
* ``exact_gemm`` -- a pure-Python brute force over ``fractions.Fraction``
  that decodes f16 through numpy's own float16 conversion.  It has no
  rounding at all and is only for tiny shapes; the tests use it to pin the C
  oracle.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from fractions import Fraction

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_gemm.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_gemm.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle_gemm.c`` with gcc into ``oracle/_build``.

    No fast-math and no fused multiply-add contraction (every product of two
    f16 values is exact in fp64 anyway, so contraction could not change a
    result; it is off so that nobody has to take that on trust)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    i64 = ctypes.c_int64
    vp = ctypes.c_void_p
    lib.oracle_f16_to_f64.restype = ctypes.c_double
    lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_gemm_f16_f64.restype = ctypes.c_int
    lib.oracle_gemm_f16_f64.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                        ctypes.c_int]
    lib.oracle_gemm_f16_f64_cells.restype = ctypes.c_int
    lib.oracle_gemm_f16_f64_cells.argtypes = [vp, vp, i64, i64, i64, i64, i64,
                                              vp, vp, i64, vp, ctypes.c_int]
    lib.oracle_threads.restype = ctypes.c_int
    lib.oracle_threads.argtypes = [ctypes.c_int]
    _lib = lib
    return lib


def _as_u16(x) -> np.ndarray:
    """View an f16 array (numpy float16 / uint16, or a CPU torch tensor) as
    its raw binary16 bit patterns, without copying when possible."""
    if hasattr(x, "detach"):  # torch tensor on the CPU
        x = x.detach().contiguous().view(dtype=__import__("torch").int16).numpy()
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16 or x.dtype == np.int16:
        return x.view(np.uint16)
    if x.dtype == np.uint16:
        return x
    raise TypeError(f"expected f16 bit patterns, got {x.dtype}")


def f16_to_f64(bits: int) -> float:
    """The oracle's own binary16 decoder (for pinning against numpy)."""
    return _load().oracle_f16_to_f64(int(bits) & 0xFFFF)


def threads(nthreads: int = 0) -> int:
    """Threads the oracle uses for a request (0 = all OpenMP allows)."""
    return _load().oracle_threads(int(nthreads))


def gemm_f64(A, B, M: int, N: int, K: int, lda: int | None = None,
             ldb: int | None = None, nthreads: int = 0) -> np.ndarray:
    """C = A.B in fp64, ascending k, as an M x N float64 array.

    ``A`` holds at least ``(M-1)*lda + K`` f16 values and ``B`` at least
    ``(K-1)*ldb + N``, row-major (flattened or 2-D)."""
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    a = _as_u16(A).reshape(-1)
    b = _as_u16(B).reshape(-1)
    if M > 0 and K > 0 and a.size < (M - 1) * lda + K:
        raise ValueError("A is smaller than M, K and lda require")
    if K > 0 and N > 0 and b.size < (K - 1) * ldb + N:
        raise ValueError("B is smaller than K, N and ldb require")
    C = np.empty((M, N), dtype=np.float64)
    if M == 0 or N == 0:
        return C
    rc = _load().oracle_gemm_f16_f64(a.ctypes.data, b.ctypes.data, C.ctypes.data,
                                     M, N, K, lda, ldb, N, int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_gemm_f16_f64 rejected its arguments")
    return C


def gemm_cells(A, B, M: int, N: int, K: int, rows, cols,
               lda: int | None = None, ldb: int | None = None,
               nthreads: int = 0) -> np.ndarray:
    """The fp64 values of the selected cells C[rows[t], cols[t]]."""
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    a = _as_u16(A).reshape(-1)
    b = _as_u16(B).reshape(-1)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != c.shape:
        raise ValueError("rows and cols differ in length")
    out = np.empty(r.size, dtype=np.float64)
    rc = _load().oracle_gemm_f16_f64_cells(a.ctypes.data, b.ctypes.data, M, N, K,
                                           lda, ldb, r.ctypes.data, c.ctypes.data,
                                           r.size, out.ctypes.data, int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_gemm_f16_f64_cells rejected its arguments")
    return out


def exact_gemm(A, B, M: int, N: int, K: int, lda: int | None = None,
               ldb: int | None = None) -> list[list[Fraction]]:
    """Brute force with exact rationals: no rounding anywhere.

    Each f16 value becomes ``Fraction(float(numpy.float16))`` -- numpy's own
    conversion, independent of the C decoder -- and every sum is exact.
    Pure-Python loops, so only for tiny shapes."""
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    a = _as_u16(A).reshape(-1).view(np.float16)
    b = _as_u16(B).reshape(-1).view(np.float16)
    fa = [Fraction(float(v)) for v in a]
    fb = [Fraction(float(v)) for v in b]
    out = []
    for i in range(M):
        row = []
        for j in range(N):
            s = Fraction(0)
            for k in range(K):
                s += fa[i * lda + k] * fb[k * ldb + j]
            row.append(s)
        out.append(row)
    return out


def grouped_gemm_f64(A, B, group_rows, E: int, M: int, N: int, K: int, C=None,
                     nthreads: int = 0) -> np.ndarray:
    """Grouped (Mixture-of-Experts) GEMM in fp64.

    The Mixture-of-Experts example of "Intel XPU Backend for Triton", section
    "Use Tensor Descriptors to load tl.dot arguments and save results": expert
    ``e`` multiplies only its first ``group_rows[e]`` token rows,
    ``A[e, :group_rows[e], :] . B[e]``; an expert with no tokens does nothing,
    and rows at or past its count are masked out, so C keeps whatever it held
    there.

    ``A`` is E x M x K and ``B`` E x K x N (f16, contiguous), ``group_rows``
    holds E integers in [0, M].  ``C`` is the output's initial contents
    (E x M x N; NaN when omitted).  Returns the E x M x N float64 result: for
    each expert, the rows below its count from ``gemm_f64`` and the others
    copied from ``C``."""
    a = _as_u16(A).reshape(E, M, K)
    b = _as_u16(B).reshape(E, K, N)
    rows = [int(r) for r in np.asarray(group_rows).reshape(-1)[:E]]
    if len(rows) != E:
        raise ValueError("group_rows holds fewer than E counts")
    out = (np.full((E, M, N), np.nan) if C is None
           else np.array(C, dtype=np.float64, copy=True).reshape(E, M, N))
    for e, m in enumerate(rows):
        if not 0 <= m <= M:
            raise ValueError(f"group_rows[{e}] = {m} is outside [0, {M}]")
        if m == 0:
            continue
        out[e, :m, :] = gemm_f64(a[e, :m, :], b[e], m, N, K, nthreads=nthreads)
    return out


# ------------------------------------------------------------------ fused epilogue

ACTIVATIONS = ("none", "relu", "leaky_relu", "gelu", "gelu_tanh", "silu")
OUT_TYPES = ("f32", "f16", "bf16")


def _erf(x: np.ndarray) -> np.ndarray:
    """erf elementwise in fp64: scipy's vectorised routine where scipy is
    installed, else the standard library's, one element at a time."""
    try:
        from scipy.special import erf
    except ImportError:
        return np.vectorize(math.erf, otypes=[np.float64])(x)
    return erf(x)


def activation_f64(x: np.ndarray, name: str, slope: float = 0.01) -> np.ndarray:
    """The activations a fused epilogue may apply, in fp64, each written from
    its mathematical definition (the pages name an ``ACTIVATION`` meta-
    parameter of the GEMM kernel -- "Intel XPU Backend for Triton", section
    "Use Proper Type Annotations" -- without fixing the set):

    * relu(x)        = x for x > 0, else 0
    * leaky_relu(x)  = x for x > 0, else slope * x
    * gelu(x)        = x * Phi(x) = x/2 * (1 + erf(x / sqrt 2))
    * gelu_tanh(x)   = x/2 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3)))
    * silu(x)        = x * sigma(x) = x / (1 + exp(-x))"""
    x = np.asarray(x, dtype=np.float64)
    if name == "none":
        return x.copy()
    if name == "relu":
        return np.where(x > 0, x, 0.0)
    if name == "leaky_relu":
        return np.where(x > 0, x, slope * x)
    if name == "gelu":
        return 0.5 * x * (1.0 + _erf(x / math.sqrt(2.0)))
    if name == "gelu_tanh":
        return 0.5 * x * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)))
    if name == "silu":
        with np.errstate(over="ignore"):
            return x / (1.0 + np.exp(-x))
    raise ValueError(f"unknown activation {name!r}")


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp64 values rounded once, to nearest with ties to even, to bfloat16
    (8 significant bits, the exponent range of binary32; subnormal spacing
    2^-133; overflow to infinity), returned as fp64.

    For |v| = m 2^e (m in [0.5, 1)) the quantum is 2^q, q = max(e - 8, -133):
    |v| / 2^q is exact in fp64 (a power-of-two scaling that stays in range),
    so rounding it to the nearest integer, ties to even, and scaling back is
    the exact round-to-nearest-even of v."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, e = np.frexp(a)
    q = np.maximum(e - 8, -133)
    y = np.ldexp(np.rint(np.ldexp(a, -q)), q)
    max_finite = (2.0 - 2.0 ** -7) * 2.0 ** 127
    y = np.where(y > max_finite, np.inf, y)
    y = np.copysign(y, x)
    special = (x == 0) | np.isnan(x) | np.isinf(x)
    return np.where(special, x, y)


def round_to_out(x: np.ndarray, out_type: str) -> np.ndarray:
    """fp64 values as the output type stores them (returned as fp64): f32 and
    f16 by numpy's conversion from fp64 (one rounding, to nearest even),
    bf16 by ``round_to_bf16``."""
    x = np.asarray(x, dtype=np.float64)
    if out_type == "f32":
        return x.astype(np.float32).astype(np.float64)
    if out_type == "f16":
        with np.errstate(over="ignore"):
            return x.astype(np.float16).astype(np.float64)
    if out_type == "bf16":
        return round_to_bf16(x)
    raise ValueError(f"unknown output type {out_type!r}")


def epilogue_f64(acc: np.ndarray, alpha: float = 1.0, bias=None, activation: str = "none",
                 slope: float = 0.01) -> np.ndarray:
    """The fused epilogue before the output rounding, in fp64:
    ``activation(alpha * acc + bias[j])`` with ``acc`` the fp64 GEMM result
    (rows x N, or batch x rows x N) and ``bias`` a length-N vector (or one per
    batch, batch x N), absent = 0."""
    v = float(alpha) * np.asarray(acc, dtype=np.float64)
    if bias is not None:
        b = np.asarray(bias, dtype=np.float64)
        v = v + (b[..., None, :] if v.ndim == 3 and b.ndim == 2 else b)
    return activation_f64(v, activation, slope)


# ------------------------------------------------------------------ row sum and GEMV

ELEM_TYPES = ("f32", "f16", "bf16")


def elements_f64(buf, elem: str) -> np.ndarray:
    """A flat buffer of f32, f16 or bf16 values (numpy array or CPU torch
    tensor, or raw bit patterns for the 16-bit types) as fp64, exactly: f32
    and f16 by numpy's conversions, bf16 as the upper half of a binary32."""
    if hasattr(buf, "detach"):
        t = buf.detach().contiguous().reshape(-1)
        import torch
        if elem == "f32":
            buf = t.view(torch.int32).numpy().view(np.float32)
        else:
            buf = t.view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(buf).reshape(-1)
    if elem == "f32":
        return a.view(np.float32).astype(np.float64) if a.dtype != np.float32 else a.astype(np.float64)
    bits = a.view(np.uint16) if a.dtype != np.uint16 else a
    if elem == "f16":
        return bits.view(np.float16).astype(np.float64)
    if elem == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(f"unknown element type {elem!r}")


def rowsum_f64(X, R: int, C: int, row_stride: int, col_stride: int, elem: str = "f16") -> np.ndarray:
    """The tiled row sum of "A Dumb Triton Runtime Error" ("The kernel
    itself"): out[r] = sum over c < C of x[r * row_stride + c * col_stride],
    every element widened exactly and the row summed with ``math.fsum`` (the
    correctly rounded fp64 sum of the exact values).  The page's tiles and
    masks (out-of-range lanes read 0, the additive identity -- section "Step 2")
    do not change this value; the tests check that separately."""
    x = elements_f64(X, elem)
    out = np.empty(R, dtype=np.float64)
    cols = np.arange(C, dtype=np.int64) * int(col_stride)
    for r in range(R):
        idx = r * int(row_stride) + cols
        if C and (idx.min() < 0 or idx.max() >= x.size):
            raise ValueError("the strided view reaches outside X")
        out[r] = math.fsum(x[idx].tolist()) if C else 0.0
    return out


def gemv_f64(A, x, M: int, K: int, lda: int | None = None, incx: int = 1) -> np.ndarray:
    """y = A . x in fp64 (f16 A: M rows of K, row stride lda; f16 x: K values
    incx apart): the GEMM oracle with N = 1 on x gathered into a column."""
    xs = _as_u16(x).reshape(-1)
    if K and (K - 1) * int(incx) >= xs.size:
        raise ValueError("x is shorter than K and incx require")
    col = np.ascontiguousarray(xs[: (K - 1) * int(incx) + 1: int(incx)] if K else xs[:0])
    return gemm_f64(A, col, M, 1, K, lda=lda, ldb=1)[:, 0]

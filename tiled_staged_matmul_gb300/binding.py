"""ctypes binding of the C ABI in ``include/tsm_gemm.h``.

Argument marshalling only: every step of the GEMM runs in ``libtsm_gemm.so``.
Importing this module loads the library and raises ``ImportError`` when it
has not been built -- there is no fallback path.

The raw functions keep the C names (``gemm_f16_f32acc`` ...) and take device
pointers as integers.  ``gemm`` and ``gemm_host`` are conveniences over torch
tensors: torch only provides the memory and the stream.
"""
from __future__ import annotations

import ctypes
import os

from .csrc import build as _build

LIB_PATH = _build.LIB_PATH

GEMM_OK = 0
GEMM_ERR_INVALID_VALUE = 1
GEMM_ERR_MISALIGNED = 2
GEMM_ERR_ALIAS = 3
GEMM_ERR_UNSUPPORTED_DEVICE = 4
GEMM_ERR_CUDA = 5
GEMM_ERR_DEVICE_TIMEOUT = 6


class GemmOptions(ctypes.Structure):
    _fields_ = [("split_k", ctypes.c_int32), ("tile_n", ctypes.c_int32),
                ("timeout_ms", ctypes.c_int32), ("inject_stall", ctypes.c_int32),
                ("tile_m", ctypes.c_int32), ("splitk_reduce", ctypes.c_int32),
                ("l2_prefetch", ctypes.c_int32), ("split_tail", ctypes.c_int32),
                ("trace", ctypes.c_void_p), ("red_cluster", ctypes.c_int32)]


ACTIVATIONS = {"none": 0, "relu": 1, "leaky_relu": 2, "gelu": 3, "gelu_tanh": 4, "silu": 5}
OUT_TYPES = {"f32": 0, "f16": 1, "bf16": 2}


class GemmEpilogue(ctypes.Structure):
    _fields_ = [("alpha", ctypes.c_float), ("bias", ctypes.c_void_p),
                ("bias_stride", ctypes.c_int64), ("activation", ctypes.c_int32),
                ("slope", ctypes.c_float), ("out_type", ctypes.c_int32)]


def epilogue(alpha=1.0, bias=0, bias_stride=0, activation="none", slope=0.01, out_type="f32"):
    """A ``GemmEpilogue``: ``activation`` and ``out_type`` by name or number,
    ``bias`` a device pointer (0 = none)."""
    act = ACTIVATIONS.get(activation, activation)
    out = OUT_TYPES.get(out_type, out_type)
    return GemmEpilogue(float(alpha), int(bias) or None, int(bias_stride), int(act), float(slope),
                        int(out))


class GemmPlanInfo(ctypes.Structure):
    _fields_ = [("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32),
                ("tile_k", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("split_k", ctypes.c_int32), ("tiles_m", ctypes.c_int32),
                ("tiles_n", ctypes.c_int32), ("k_blocks", ctypes.c_int32),
                ("units", ctypes.c_int64), ("grid", ctypes.c_int32),
                ("group_m", ctypes.c_int32), ("stage_bytes", ctypes.c_int64),
                ("smem_bytes", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
                ("fused_reduce", ctypes.c_int32), ("tail_tiles", ctypes.c_int32),
                ("tail_split", ctypes.c_int32), ("tail_narrow", ctypes.c_int32),
                ("red_cluster", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class GemmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{gemm_status_string(status)}: {message}")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    lib.gemm_f16_f32acc.restype = ctypes.c_int
    lib.gemm_f16_f32acc.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, vp]
    lib.gemm_f16_f32acc_batched.restype = ctypes.c_int
    lib.gemm_f16_f32acc_batched.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                            i64, i64, i64, i64, vp]
    lib.gemm_f16_f32acc_opts.restype = ctypes.c_int
    lib.gemm_f16_f32acc_opts.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                         i64, i64, i64, i64, ctypes.POINTER(GemmOptions), vp]
    lib.gemm_plan.restype = ctypes.c_int
    lib.gemm_plan.argtypes = [i64, i64, i64, i64, ctypes.POINTER(GemmOptions), i32,
                              ctypes.POINTER(GemmPlanInfo)]
    lib.gemm_plan_grouped.restype = ctypes.c_int
    lib.gemm_plan_grouped.argtypes = [i64, i64, i64, i64, ctypes.POINTER(GemmOptions), i32,
                                      ctypes.POINTER(GemmPlanInfo)]
    lib.gemm_get_device_status.restype = ctypes.c_int
    lib.gemm_get_device_status.argtypes = [vp]
    lib.gemm_last_error_string.restype = ctypes.c_char_p
    lib.gemm_last_error_string.argtypes = []
    lib.gemm_status_string.restype = ctypes.c_char_p
    lib.gemm_status_string.argtypes = [ctypes.c_int]
    lib.gemm_version.restype = ctypes.c_int32
    lib.gemm_version.argtypes = []
    lib.gemm_f16_f32acc_grouped.restype = ctypes.c_int
    lib.gemm_f16_f32acc_grouped.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64,
                                            i64, i64, i64, vp]
    lib.gemm_f16_f32acc_grouped_opts.restype = ctypes.c_int
    lib.gemm_f16_f32acc_grouped_opts.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                                 i64, i64, i64, i64, ctypes.POINTER(GemmOptions),
                                                 vp]
    lib.gemm_f16_fused.restype = ctypes.c_int
    lib.gemm_f16_fused.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, i64, i64, i64,
                                   ctypes.POINTER(GemmEpilogue), ctypes.POINTER(GemmOptions), vp]
    lib.gemm_f16_grouped_fused.restype = ctypes.c_int
    lib.gemm_f16_grouped_fused.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, i64,
                                           i64, i64, ctypes.POINTER(GemmEpilogue),
                                           ctypes.POINTER(GemmOptions), vp]
    lib.rowsum_f32acc.restype = ctypes.c_int
    lib.rowsum_f32acc.argtypes = [vp, i32, vp, i64, i64, i64, i64, vp]
    lib.gemv_f16_f32acc.restype = ctypes.c_int
    lib.gemv_f16_f32acc.argtypes = [vp, vp, vp, i64, i64, i64, i64, vp]
    lib.gemm_f16_f32acc_splitk_noalloc.restype = ctypes.c_int
    lib.gemm_f16_f32acc_splitk_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                                   i32, vp]
    return lib


_lib = _load()


def _opts(split_k=0, tile_n=0, timeout_ms=0, inject_stall=0, tile_m=0, splitk_reduce=0):
    return GemmOptions(int(split_k), int(tile_n), int(timeout_ms), int(inject_stall), int(tile_m),
                       int(splitk_reduce))


# ------------------------------------------------------------------ raw C names

def gemm_f16_f32acc(A, B, C, M, N, K, lda, ldb, ldc, stream=0) -> int:
    return _lib.gemm_f16_f32acc(A, B, C, M, N, K, lda, ldb, ldc, stream)


def gemm_f16_f32acc_batched(A, B, C, M, N, K, lda, ldb, ldc, strideA, strideB, strideC,
                            batch, stream=0) -> int:
    return _lib.gemm_f16_f32acc_batched(A, B, C, M, N, K, lda, ldb, ldc, strideA, strideB,
                                        strideC, batch, stream)


def gemm_f16_f32acc_opts(A, B, C, M, N, K, lda, ldb, ldc, strideA, strideB, strideC, batch,
                         opts: GemmOptions | None = None, stream=0) -> int:
    p = ctypes.byref(opts) if opts is not None else None
    return _lib.gemm_f16_f32acc_opts(A, B, C, M, N, K, lda, ldb, ldc, strideA, strideB,
                                     strideC, batch, p, stream)


def gemm_f16_f32acc_grouped(A, B, C, group_rows, groups, M, N, K, lda, ldb, ldc, strideA,
                            strideB, strideC, stream=0) -> int:
    return _lib.gemm_f16_f32acc_grouped(A, B, C, group_rows, groups, M, N, K, lda, ldb, ldc,
                                        strideA, strideB, strideC, stream)


def gemm_f16_f32acc_grouped_opts(A, B, C, group_rows, groups, M, N, K, lda, ldb, ldc, strideA,
                                 strideB, strideC, opts: GemmOptions | None = None,
                                 stream=0) -> int:
    p = ctypes.byref(opts) if opts is not None else None
    return _lib.gemm_f16_f32acc_grouped_opts(A, B, C, group_rows, groups, M, N, K, lda, ldb, ldc,
                                             strideA, strideB, strideC, p, stream)


def gemm_f16_fused(A, B, C, M, N, K, lda, ldb, ldc, strideA, strideB, strideC, batch,
                   epi: GemmEpilogue | None = None, opts: GemmOptions | None = None,
                   stream=0) -> int:
    e = ctypes.byref(epi) if epi is not None else None
    o = ctypes.byref(opts) if opts is not None else None
    return _lib.gemm_f16_fused(A, B, C, M, N, K, lda, ldb, ldc, strideA, strideB, strideC, batch,
                               e, o, stream)


def gemm_f16_grouped_fused(A, B, C, group_rows, groups, M, N, K, lda, ldb, ldc, strideA, strideB,
                           strideC, epi: GemmEpilogue | None = None,
                           opts: GemmOptions | None = None, stream=0) -> int:
    e = ctypes.byref(epi) if epi is not None else None
    o = ctypes.byref(opts) if opts is not None else None
    return _lib.gemm_f16_grouped_fused(A, B, C, group_rows, groups, M, N, K, lda, ldb, ldc, strideA,
                                       strideB, strideC, e, o, stream)


def rowsum_f32acc(X, elem_type, out, R, C, row_stride, col_stride, stream=0) -> int:
    return _lib.rowsum_f32acc(X, OUT_TYPES.get(elem_type, elem_type), out, R, C, row_stride,
                              col_stride, stream)


def gemv_f16_f32acc(A, x, y, M, K, lda, incx=1, stream=0) -> int:
    return _lib.gemv_f16_f32acc(A, x, y, M, K, lda, incx, stream)


def gemm_f16_f32acc_splitk_noalloc(A, B, C, M, N, K, lda, ldb, ldc, split_k=0, stream=0) -> int:
    """The entry point that allocates nothing (split-K partials in a fixed
    16 MiB device array inside the library); see include/tsm_gemm.h."""
    return _lib.gemm_f16_f32acc_splitk_noalloc(A, B, C, M, N, K, lda, ldb, ldc, split_k, stream)


def gemm_plan(M, N, K, batch=1, opts: GemmOptions | None = None, num_sms=0) -> dict:
    info = GemmPlanInfo()
    p = ctypes.byref(opts) if opts is not None else None
    st = _lib.gemm_plan(M, N, K, batch, p, num_sms, ctypes.byref(info))
    if st != GEMM_OK:
        raise GemmError(st, gemm_last_error_string())
    return info.as_dict()


def gemm_plan_grouped(M, N, K, groups=1, opts: GemmOptions | None = None, num_sms=0) -> dict:
    info = GemmPlanInfo()
    p = ctypes.byref(opts) if opts is not None else None
    st = _lib.gemm_plan_grouped(M, N, K, groups, p, num_sms, ctypes.byref(info))
    if st != GEMM_OK:
        raise GemmError(st, gemm_last_error_string())
    return info.as_dict()


def gemm_get_device_status(stream=0) -> int:
    return _lib.gemm_get_device_status(stream)


def gemm_last_error_string() -> str:
    return _lib.gemm_last_error_string().decode()


def gemm_status_string(status: int) -> str:
    return _lib.gemm_status_string(int(status)).decode()


def gemm_version() -> int:
    return _lib.gemm_version()


def check(status: int) -> None:
    if status != GEMM_OK:
        raise GemmError(status, gemm_last_error_string())


# ------------------------------------------------------------------ torch conveniences

def _stream_handle(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def gemm(A, B, out=None, *, alpha=1.0, bias=None, activation="none", slope=0.01, out_dtype=None,
         split_k=0, tile_n=0, tile_m=0, timeout_ms=0, inject_stall=0, stream=None):
    """``out = activation(alpha * (A @ B) + bias)`` for f16 CUDA tensors A
    (M x K) and B (K x N); ``out`` is f32 unless ``out_dtype`` (or the given
    ``out``) says torch.float16 / torch.bfloat16.

    3-D tensors (batch x M x K, batch x K x N) run as one batched call;
    ``bias`` is an f32 CUDA tensor of N values (or batch x N).  Rows may be
    padded (``stride(-2) >= size(-1)``) but the last stride must be 1.
    Returns ``out`` (allocated with ``torch.empty`` when not given)."""
    import torch
    if A.dtype != torch.float16 or B.dtype != torch.float16:
        raise TypeError("A and B must be torch.float16")
    batched = A.dim() == 3
    if A.dim() != B.dim() or A.dim() not in (2, 3):
        raise ValueError("A and B must both be 2-D or both 3-D")
    M, K = A.shape[-2], A.shape[-1]
    K2, N = B.shape[-2], B.shape[-1]
    if K != K2:
        raise ValueError(f"inner sizes differ: {K} vs {K2}")
    batch = A.shape[0] if batched else 1
    if batched and B.shape[0] != batch:
        raise ValueError("batch sizes differ")
    dtype = out.dtype if out is not None else (out_dtype or torch.float32)
    out_names = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}
    if dtype not in out_names:
        raise TypeError("out must be torch.float32, torch.float16 or torch.bfloat16")
    if out is None:
        # rows padded to a 16-byte pitch (the TMA's rule); the view hides it
        per16 = 16 // torch.tensor([], dtype=dtype).element_size()
        ldc_alloc = max(per16, -(-N // per16) * per16)
        shape = (batch, M, ldc_alloc) if batched else (M, ldc_alloc)
        out = torch.empty(shape, dtype=dtype, device=A.device)[..., :N]
    for t, name in ((A, "A"), (B, "B"), (out, "out")):
        if t.numel() and t.stride(-1) != 1:
            raise ValueError(f"{name} must have a unit last stride")
    # Any row pitch works; pitches that are not multiples of 16 bytes (and
    # unaligned bases) cost the library a repacking copy.
    lda = A.stride(-2) if M > 1 else max(K, 1)
    ldb = B.stride(-2) if K > 1 else max(N, 1)
    ldc = out.stride(-2) if M > 1 else max(N, 1)
    sA = A.stride(0) if batched else 0
    sB = B.stride(0) if batched else 0
    sC = out.stride(0) if batched else 0
    opts = _opts(split_k, tile_n, timeout_ms, inject_stall, tile_m)
    if bias is not None:
        if bias.dtype != torch.float32 or not bias.is_cuda or bias.shape[-1] != N:
            raise ValueError("bias must be a CUDA float32 tensor of N values (or batch x N)")
        if bias.stride(-1) != 1:
            raise ValueError("bias must have a unit last stride")
    epi = epilogue(alpha, bias.data_ptr() if bias is not None else 0,
                   bias.stride(0) if bias is not None and bias.dim() == 2 else 0,
                   activation, slope, out_names[dtype])
    st = gemm_f16_fused(A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N, K, lda, ldb, ldc, sA, sB,
                        sC, batch, epi, opts, _stream_handle(stream))
    check(st)
    return out


def grouped_gemm(A, B, group_rows, out=None, *, alpha=1.0, bias=None, activation="none",
                 slope=0.01, out_dtype=None, tile_n=0, tile_m=0, stream=None):
    """Grouped (Mixture-of-Experts) GEMM on CUDA tensors: for each group g,
    ``out[g, :group_rows[g]] = A[g, :group_rows[g]] @ B[g]``.

    A is groups x M x K and B groups x K x N (f16), ``group_rows`` a CUDA
    int32 tensor of ``groups`` row counts in [0, M].  Rows at or past a
    group's count keep the contents of ``out`` (zeros when ``out`` is not
    given).  Returns ``out`` (groups x M x N, f32)."""
    import torch
    if A.dtype != torch.float16 or B.dtype != torch.float16:
        raise TypeError("A and B must be torch.float16")
    if A.dim() != 3 or B.dim() != 3 or A.shape[0] != B.shape[0] or A.shape[2] != B.shape[1]:
        raise ValueError("A must be G x M x K and B G x K x N")
    if group_rows.dtype != torch.int32 or not group_rows.is_cuda or group_rows.numel() != A.shape[0]:
        raise ValueError("group_rows must be a CUDA int32 tensor of one count per group")
    G, M, K = A.shape
    N = B.shape[2]
    dtype = out.dtype if out is not None else (out_dtype or torch.float32)
    out_names = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}
    if dtype not in out_names:
        raise TypeError("out must be torch.float32, torch.float16 or torch.bfloat16")
    if out is None:
        per16 = 16 // torch.tensor([], dtype=dtype).element_size()
        ldc_alloc = max(per16, -(-N // per16) * per16)
        out = torch.zeros((G, M, ldc_alloc), dtype=dtype, device=A.device)[..., :N]
    if tuple(out.shape) != (G, M, N):
        raise ValueError("out must be a G x M x N tensor")
    for t, name in ((A, "A"), (B, "B"), (out, "out")):
        if t.numel() and t.stride(-1) != 1:
            raise ValueError(f"{name} must have a unit last stride")
    rows = group_rows.contiguous()
    opts = _opts(0, tile_n, 0, 0, tile_m)
    if bias is not None and (bias.dtype != torch.float32 or not bias.is_cuda
                             or bias.shape[-1] != N or bias.stride(-1) != 1):
        raise ValueError("bias must be a CUDA float32 tensor of N values (or groups x N)")
    epi = epilogue(alpha, bias.data_ptr() if bias is not None else 0,
                   bias.stride(0) if bias is not None and bias.dim() == 2 else 0,
                   activation, slope, out_names[dtype])
    st = gemm_f16_grouped_fused(A.data_ptr(), B.data_ptr(), out.data_ptr(), rows.data_ptr(),
                                G, M, N, K, A.stride(1), B.stride(1), out.stride(1),
                                A.stride(0), B.stride(0), out.stride(0), epi, opts,
                                _stream_handle(stream))
    check(st)
    return out


def rowsum(X, out=None, *, stream=None):
    """Row sums of a 2-D CUDA tensor (f32, f16 or bf16; any strides): an f32
    tensor of X.shape[0] values, summed in f32 in a fixed order."""
    import torch
    names = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}
    if X.dtype not in names or X.dim() != 2 or not X.is_cuda:
        raise ValueError("X must be a 2-D CUDA tensor of float32, float16 or bfloat16")
    R, C = X.shape
    if out is None:
        out = torch.empty(R, dtype=torch.float32, device=X.device)
    if out.dtype != torch.float32 or out.numel() != R or (R and out.stride(0) != 1):
        raise ValueError("out must be a contiguous float32 tensor of X.shape[0] values")
    check(rowsum_f32acc(X.data_ptr(), names[X.dtype], out.data_ptr(), R, C, X.stride(0),
                        X.stride(1), _stream_handle(stream)))
    return out


def gemv(A, x, out=None, *, stream=None):
    """``A @ x`` for an f16 CUDA matrix A (unit last stride) and f16 vector x
    (any stride): an f32 vector."""
    import torch
    if A.dtype != torch.float16 or x.dtype != torch.float16 or A.dim() != 2 or x.dim() != 1:
        raise ValueError("A must be a 2-D and x a 1-D torch.float16 CUDA tensor")
    M, K = A.shape
    if x.numel() != K:
        raise ValueError("x must hold A.shape[1] values")
    if K and A.stride(1) != 1:
        raise ValueError("A must have a unit last stride")
    if out is None:
        out = torch.empty(M, dtype=torch.float32, device=A.device)
    check(gemv_f16_f32acc(A.data_ptr(), x.data_ptr(), out.data_ptr(), M, K,
                          A.stride(0) if M > 1 else max(K, 1), x.stride(0) if K > 1 else 1,
                          _stream_handle(stream)))
    return out


def gemm_host(A_host, B_host, C_host, dA, dB, dC, stream=None):
    """End-to-end call from host memory: copy A and B (pinned CPU f16
    tensors) into the device buffers dA and dB, run the GEMM into dC, copy dC
    back into C_host (pinned CPU f32).  All on one stream, asynchronously;
    synchronise the stream before reading C_host."""
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    with torch.cuda.stream(s):
        dA.copy_(A_host, non_blocking=True)
        dB.copy_(B_host, non_blocking=True)
        gemm(dA, dB, dC, stream=s)
        C_host.copy_(dC, non_blocking=True)
    return C_host


class HostPipeline:
    """C = A . B for a stream of host-resident problems of one shape.

    Each ``submit`` copies A and B (pinned CPU f16 tensors) to the device,
    runs the GEMM and copies C back into the given pinned CPU f32 tensor.
    ``depth`` device buffer sets and three CUDA streams (upload, GEMM,
    download) let the upload of one problem overlap the GEMM and the download
    of the previous ones; events order the three stages of each problem and
    keep a buffer set from being reused before its result has been read back.
    Torch provides the memory, streams and copies; the GEMM is this library's.
    Call ``synchronize`` before reading the last ``depth`` results."""

    def __init__(self, M, N, K, depth=2, device=None):
        import torch
        self.M, self.N, self.K, self.depth = M, N, K, depth
        dev = torch.device("cuda") if device is None else torch.device(device)
        self.dA = [torch.empty((M, K), dtype=torch.float16, device=dev) for _ in range(depth)]
        self.dB = [torch.empty((K, N), dtype=torch.float16, device=dev) for _ in range(depth)]
        ldc = max(4, -(-N // 4) * 4)
        self.dC = [torch.empty((M, ldc), dtype=torch.float32, device=dev)[:, :N]
                   for _ in range(depth)]
        self.s_in = torch.cuda.Stream(device=dev)
        self.s_gemm = torch.cuda.Stream(device=dev)
        self.s_out = torch.cuda.Stream(device=dev)
        self.in_done = [torch.cuda.Event() for _ in range(depth)]
        self.gemm_done = [torch.cuda.Event() for _ in range(depth)]
        self.out_done = [torch.cuda.Event() for _ in range(depth)]
        self.used = [False] * depth
        self.count = 0

    def submit(self, A_host, B_host, C_host):
        import torch
        i = self.count % self.depth
        self.count += 1
        if self.used[i]:
            self.s_in.wait_event(self.out_done[i])  # buffer set i is free again
        with torch.cuda.stream(self.s_in):
            self.dA[i].copy_(A_host, non_blocking=True)
            self.dB[i].copy_(B_host, non_blocking=True)
            self.in_done[i].record(self.s_in)
        self.s_gemm.wait_event(self.in_done[i])
        gemm(self.dA[i], self.dB[i], self.dC[i], stream=self.s_gemm)
        self.gemm_done[i].record(self.s_gemm)
        self.s_out.wait_event(self.gemm_done[i])
        with torch.cuda.stream(self.s_out):
            C_host.copy_(self.dC[i], non_blocking=True)
            self.out_done[i].record(self.s_out)
        self.used[i] = True
        return C_host

    def synchronize(self):
        self.s_out.synchronize()

"""Cases for the serialised-run determinism test, runnable on their own.

    python tests/serial_cases.py OUT.pt

runs every case below through the C ABI and saves each C (CPU f32) to
OUT.pt.  The test runs this file in a child process with
CUDA_LAUNCH_BLOCKING=1 -- every launch then waits for the previous one to
finish, so no two kernels, copies or memsets overlap -- and compares with the
same cases run in its own process without it: the split-K sums (in the
kernel, in clusters, in a second kernel, over a partial last wave), the
256 x 512 tile's single accumulator handed from tile to tile, and the
grouped call must not depend on how the GPU happened to schedule the work."""
from __future__ import annotations

import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# (name, M, N, K, options as GemmOptions fields, batch)
CASES = [
    ("split_in_kernel", 256, 256, 65536, {"red_cluster": 1}, 1),
    ("split_cluster4", 256, 256, 65536, {"red_cluster": 4}, 1),
    ("split_cluster2", 300, 250, 30000, {"red_cluster": 2, "split_k": 16, "tile_m": 128,
                                         "tile_n": 256}, 1),
    ("split_separate", 256, 256, 65536, {"splitk_reduce": 1}, 1),
    ("split_pairs", 512, 512, 32768, {"tile_m": 256, "tile_n": 256}, 1),
    ("k_range_tail", 4096, 4096, 1024, {"split_tail": 1}, 1),
    ("column_slice_tail", 2304, 2304, 512, {"split_tail": 3}, 1),
    ("batched_split", 200, 136, 12000, {}, 3),
    ("wide_pair_tile", 4096, 4096, 512, {"tile_m": 256, "tile_n": 512}, 1),
]
GROUPED = ("grouped", 6, 300, 256, 1024, [300, 0, 129, 17, 256, 1])


def run_all() -> dict:
    from tiled_staged_matmul_gb300 import binding as b, synthetic
    s = torch.cuda.current_stream().cuda_stream
    out = {}
    for name, M, N, K, fields, batch in CASES:
        A, B = synthetic.operands(M, N, K, "uniform", seed=M + N + K, batch=batch)
        dA, dB = A.cuda().contiguous(), B.cuda().contiguous()
        C = torch.empty((batch, M, N) if batch > 1 else (M, N), dtype=torch.float32, device="cuda")
        o = b.GemmOptions()
        for k, v in fields.items():
            setattr(o, k, v)
        b.check(b.gemm_f16_f32acc_opts(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, K, N, N,
                                       M * K if batch > 1 else 0, K * N if batch > 1 else 0,
                                       M * N if batch > 1 else 0, batch, o, s))
        b.check(b.gemm_get_device_status(s))
        out[name] = C.cpu()
    name, G, M, N, K, rows = GROUPED
    A, B = synthetic.operands(M, N, K, "uniform", seed=G + M, batch=G)
    dA, dB = A.cuda().contiguous(), B.cuda().contiguous()
    C = torch.zeros((G, M, N), dtype=torch.float32, device="cuda")
    counts = torch.tensor(rows, dtype=torch.int32, device="cuda")
    b.check(b.gemm_f16_f32acc_grouped(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), counts.data_ptr(),
                                      G, M, N, K, K, N, N, M * K, K * N, M * N, s))
    b.check(b.gemm_get_device_status(s))
    out[name] = C.cpu()
    return out


if __name__ == "__main__":
    torch.save(run_all(), sys.argv[1])

#!/usr/bin/env python3
"""Throughput of the GB300 f16 x f16 -> f32 GEMM, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline] [--no-e2e]

A step is one call of the C ABI's GEMM on one synthetic, seeded workload
(default: 8192 x 8192 x 8192, f16 N(0, 1/sqrt(K)) operands), inputs resident
in HBM.  Each step is timed with CUDA events on the launching stream; the K
steps sit between a barrier + device synchronisation on both sides and the
slowest rank decides.  With N > 1 every rank runs an independent replica
(the GEMM is single-GPU; the value is the sum over ranks: weak scaling).

``--impl reference`` times the CPU oracle (fp64 triple loop) instead, on a
bounded row sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "gemm_8192x8192x8192_normal_invsqrtk"
METRIC = "GEMM TFLOP/s (f16 in, f32 acc) and % of GB300 dense-f16 / HBM roofline"
L2_BYTES = 129 * 1024 * 1024
# The kernels and the host code that plans their launches: recorded DRAM
# traffic is valid only for the exact code that produced it.
KERNEL_SOURCES = ["tiled_staged_matmul_gb300/csrc/gemm_kernels.cu",
                  "tiled_staged_matmul_gb300/csrc/gemm_kernel.cuh",
                  "tiled_staged_matmul_gb300/csrc/gemm_epi.cu",
                  "tiled_staged_matmul_gb300/csrc/rowsum_kernels.cu",
                  "tiled_staged_matmul_gb300/csrc/gemm_internal.h",
                  "tiled_staged_matmul_gb300/csrc/ptx.cuh",
                  "tiled_staged_matmul_gb300/csrc/gemm_api.cu"]


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--warm-seconds", type=float, default=0.5,
                   help="after the warm-up steps, keep warming up until the GPU has been busy this long")
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD,
                   help="one of the named workloads in tiled_staged_matmul_gb300.synthetic "
                        "(WORKLOADS, or GROUPED_WORKLOADS for the grouped call)")
    p.add_argument("--shape", default=None,
                   help="MxNxK: an ad-hoc shape with N(0, 1/sqrt(K)) operands instead of --workload")
    p.add_argument("--tile-m", type=int, default=0, help="128 or 256 (CTA pair); 0: planner")
    p.add_argument("--tile-n", type=int, default=0, help="64, 128, 256 or 512; 0: planner")
    p.add_argument("--split-k", type=int, default=0, help="K ranges; 0: planner")
    p.add_argument("--splitk-reduce", type=int, default=0,
                   help="0/2: in-kernel split-K sum when possible, 1: separate reduce kernel")
    p.add_argument("--red-cluster", type=int, default=0,
                   help="in-kernel split-K sum taken in clusters of 2 or 4 CTAs; 1: off; 0: planner")
    p.add_argument("--ld-pad", type=int, default=0,
                   help="lay A, B and C out with lda = K + p, ldb = ldc = N + p elements; an odd p "
                        "makes every operand unaddressable by the TMA (the repacking path)")
    p.add_argument("--act", default="none",
                   help="fused epilogue activation: none, relu, leaky_relu, gelu, gelu_tanh, silu")
    p.add_argument("--bias", action="store_true", help="fused epilogue: add a per-column f32 bias")
    p.add_argument("--out", default="f32", choices=("f32", "f16", "bf16"),
                   help="fused epilogue: the element type of C")
    p.add_argument("--trace", action="store_true",
                   help="add a per-CTA phase timeline (one extra traced step) to the JSON line")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip timing the other four GEMM shapes beside the default line")
    p.add_argument("--workload-rounds", type=int, default=100,
                   help="interleaved rounds (one step of each shape) timed for the workloads table")
    p.add_argument("--e2e-steps", type=int, default=30,
                   help="end-to-end steps timed (the three-deep pipeline fills and drains once)")
    return p.parse_args(argv)


# ------------------------------------------------------------------ distributed helpers

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(flops_per_rank: float, ms_local: float, world: int, device=None):
    """Whole-job throughput of `world` independent replicas: every rank did
    `flops_per_rank`; the slowest rank's time per step decides.  Returns
    (TFLOP/s over all ranks, the max ms per step)."""
    ms = max_over_ranks(ms_local, world, device)
    return world * flops_per_rank / (ms * 1e-3) / 1e12, ms


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ peaks and roofline

def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the GEMM kernel from an ncu capture, if one
    was recorded for exactly the current kernel source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if e and e.get("kernel_hash") == kernel_source_hash():
        return e.get("dram_bytes_per_launch")
    return None


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampled every 20 ms in the background; samples are kept
    with their host time so that only those inside the timed region count."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    # nvidia-smi's readings refresh about every 0.1 s and describe the time
    # before the reading: a state of the timed region shows up to LAG_S later.
    LAG_S = 0.25

    def summary(self, t0: float, t1: float) -> dict:
        """SM clock (median) and throttle reasons of the timed region
        [t0, t1]: the clock from readings taken in the region shifted by
        0.1 s, the reasons from every reading up to LAG_S after it."""
        def window(a, b):
            return [s for (t, s) in self.samples if a <= t <= b]
        rows = window(t0 + 0.1, t1 + 0.1)
        if not rows:  # region shorter than the sampling period: nearest samples
            rows = [s for (t, s) in sorted(self.samples, key=lambda ts: abs(ts[0] - (t0 + t1) / 2))[:3]]
        reason_rows = window(t0, t1 + self.LAG_S) or rows
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
        for r in reason_rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 8:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------------ our arm

def timed_loop(args, call, flush, stream, world, local_rank):
    """W untimed warm-up steps, then K steps each bracketed by CUDA events on
    the launching stream (L2 flushed before every step when ``flush`` is
    given), a barrier and a device synchronisation on both sides, SM clocks
    sampled throughout.  Returns (ms per step, wall start, wall end, sampler)."""
    import torch
    from tiled_staged_matmul_gb300 import binding
    # The sampler runs from the first warm-up step on: the timed steps follow
    # the warm-up with no idle gap, in the clock and power state the workload
    # has settled in, whatever the number of steps.
    sampler = ClockSampler(local_rank)
    sampler.start()
    for _ in range(max(args.warmup, 3)):
        if flush:
            flush()
        call()
    # The burst regime: 30 steps before the power cap can engage (~0.1 s of
    # load on GB300), reported beside the line, not as it.
    torch.cuda.synchronize()
    b_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(30)]
    for e0, e1 in b_ev:
        if flush:
            flush()
        e0.record(stream)
        call()
        e1.record(stream)
    torch.cuda.synchronize()
    burst_ms = sum(e0.elapsed_time(e1) for e0, e1 in b_ev) / len(b_ev)
    # ... and on until the GPU has been loaded for warm_seconds, so that the
    # timed steps run in the clock and power state the workload settles in
    # (on GB300 the power cap lowers the SM clock ~0.1 s into a dense GEMM).
    torch.cuda.synchronize()
    w0 = time.time()
    while time.time() - w0 < args.warm_seconds:
        for _ in range(8):
            if flush:
                flush()
            call()
        torch.cuda.synchronize()
    binding.check(binding.gemm_get_device_status(stream.cuda_stream))
    torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(args.steps):
        if flush:
            flush()
        starts[i].record(stream)
        call()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    time.sleep(ClockSampler.LAG_S + 0.1)  # readings trail the GPU's state
    sampler.stop()
    binding.check(binding.gemm_get_device_status(stream.cuda_stream))
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], t0, t1, sampler, burst_ms


def step_stats(per_step_ms):
    """Mean, median and minimum of the per-step event times (ms)."""
    return {"mean": round(statistics.fmean(per_step_ms), 5),
            "median": round(statistics.median(per_step_ms), 5),
            "min": round(min(per_step_ms), 5)}


def burst_of(flops, algorithmic_bytes, ms):
    """The first 30 steps after the minimum warm-up, before the power cap can
    engage, against the burst peaks (reported beside the line)."""
    r = roofline_of(flops, algorithmic_bytes, ms, None, "",
                    {"sm_mhz": None, "sm_max_mhz": None, "reasons": []})
    return {"steps": 30, "ms_per_step": round(ms, 5), "value": round(flops / (ms * 1e-3) / 1e12, 2),
            "unit": "TFLOP/s", "roofline_frac": r["frac"], "bound": r["bound"], "peak": r["peak"]}


def power_capped(clocks) -> bool:
    """The timed region ran under the power cap (or well below the maximum
    SM clock): the sustained regime."""
    if not clocks:
        return False
    if "sw_power_cap" in clocks.get("reasons", []):
        return True
    sm, smax = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    return bool(sm and smax and sm < 0.97 * smax)


def roofline_of(flops, algorithmic_bytes, ms, traffic, kernel, clocks=None):
    """Achieved against the slower of the two roofs: dense tensor peak for
    the flops, HBM bandwidth for the algorithmic bytes (both measured).  The
    tensor peak is the burst one, or the sustained one (cuBLAS back to back
    for seconds, under the power cap) when the timed region ran power-capped."""
    peaks = measured_peaks()
    tflops_launch = flops / (ms * 1e-3) / 1e12
    gbs_launch = algorithmic_bytes / (ms * 1e-3) / 1e9
    t_tensor = flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = algorithmic_bytes / (peaks["hbm_gbs"] * 1e9)
    sustained = power_capped(clocks) and peaks.get("bf16_tflops_sustained")
    tensor_peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    if t_tensor >= t_hbm:
        roofline = {"bound": "tensor", "achieved": round(tflops_launch, 2),
                    "peak": tensor_peak, "unit": "TFLOP/s",
                    "frac": round(tflops_launch / tensor_peak, 4)}
    else:
        roofline = {"bound": "hbm", "achieved": round(gbs_launch, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(gbs_launch / peaks["hbm_gbs"], 4)}
    roofline["traffic"] = traffic
    roofline["peak_source"] = (f"{peaks['source']} (MEASURED_PEAKS.json bf16 "
                               f"{'sustained: the timed region ran power-capped' if sustained else 'burst'}"
                               "; f16 dense rate taken equal to bf16, the nominal ratio)"
                               if roofline["bound"] == "tensor" else
                               f"{peaks['source']} (MEASURED_PEAKS.json copy bandwidth)")
    roofline["kernel"] = kernel
    if roofline["bound"] == "tensor":
        roofline["per_clock"] = per_clock_peak(tflops_launch, clocks)
    return roofline


# Dense f16 tensor rate per SM and clock assumed for the secondary peak
# (B200's published dense figure divided by its SMs and clock).
F16_FLOP_PER_CLK_PER_SM = 8192


def per_clock_peak(tflops, clocks, sms=None):
    """The secondary tensor peak: SMs x 8192 dense f16 flop per clock x SM
    clock, at the maximum clock and at the median clock the timed region ran
    at, with the achieved rate's fraction of each (SMs: the current device's
    unless given)."""
    if sms is None:
        import torch
        if not torch.cuda.is_available():
            return None
        sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    out = {"sms": sms, "flop_per_clk_per_sm": F16_FLOP_PER_CLK_PER_SM}
    for key, mhz in (("at_max_clock", (clocks or {}).get("sm_max_mhz")),
                     ("at_load_clock", (clocks or {}).get("sm_mhz"))):
        if mhz:
            peak = sms * F16_FLOP_PER_CLK_PER_SM * mhz * 1e6 / 1e12
            out[key] = {"mhz": mhz, "tflops": round(peak, 1), "frac": round(tflops / peak, 4)}
    return out


def run_grouped(args, rank, local_rank, world):
    """A grouped (Mixture-of-Experts) workload: one step is one grouped call
    over every expert's routed rows; the metric counts the flops of those
    rows only (2 x rows x N x K summed over the experts)."""
    import torch
    from tiled_staged_matmul_gb300 import binding, synthetic

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = synthetic.GROUPED_WORKLOADS[args.workload]
    A_h, B_h = synthetic.grouped_operands(w)
    counts_h = w.counts()
    A, B, counts = A_h.to(dev), B_h.to(dev), counts_h.to(dev)
    C = torch.empty((w.groups, w.M, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    opts = binding.GemmOptions(0, args.tile_n, 0, 0, args.tile_m)
    per_launch = min(w.groups, 256)
    plan = binding.gemm_plan_grouped(w.M, w.N, w.K, per_launch, binding.GemmOptions(0, args.tile_n, 0, 0,
                                                                                    args.tile_m))
    launches_per_call = -(-w.groups // 256)
    flops = w.flops(counts_h)
    abytes = w.algorithmic_bytes(counts_h)
    working_set = 2 * A.numel() + 2 * B.numel() + 4 * C.numel()
    flush = working_set < 2 * L2_BYTES
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    sweep = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    sink = torch.empty(1, dtype=torch.float32, device=dev) if flush else None

    def flush_l2():
        scrub.zero_()
        torch.sum(sweep, dim=0, keepdim=True, out=sink)

    def call():
        binding.check(binding.gemm_f16_f32acc_grouped_opts(
            A.data_ptr(), B.data_ptr(), C.data_ptr(), counts.data_ptr(), w.groups, w.M, w.N, w.K,
            w.K, w.N, w.N, w.M * w.K, w.K * w.N, w.M * w.N, opts, stream.cuda_stream))

    per_step_ms, t0, t1, sampler, burst_ms = timed_loop(args, call, flush_l2 if flush else None,
                                                        stream, world, local_rank)
    ms_local = sum(per_step_ms) / len(per_step_ms)
    clocks = sampler.summary(t0, t1)
    value, ms = replica_throughput(flops, ms_local, world, dev)
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": w.name, "groups": w.groups, "M": w.M, "N": w.N, "K": w.K,
                   "routed_rows": int(counts_h.sum()), "tokens": w.tokens, "dist": w.dist,
                   "seed": w.seed, "accumulate": "f32", "tile_m": plan["tile_m"],
                   "tile_n": plan["tile_n"], "split_k": 1, "stages": plan["stages"],
                   "grid": plan["grid"],
                   "l2": "flushed before every step (write 2xL2, then read 2xL2)" if flush else
                         f"inputs+output {working_set / 2**20:.0f} MiB > L2, no flush",
                   "parallelism": f"replicas x{world}"},
        "gpu_launches": args.steps * launches_per_call,
        "roofline": roofline_of(flops, abytes, ms_local, recorded_traffic(w.name),
                                "tsm_gemm_tcgen05_kernel (grouped)", clocks),
        "burst": burst_of(flops, abytes, burst_ms),
    }
    result["clocks"] = {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = grouped_cpu_baseline(w, A_h, B_h, counts_h, target_s=15.0)
    return result


def run_rows(args, rank, local_rank, world):
    """A row-sum or GEMV workload: one step is one call over the whole matrix;
    the metric counts one add (row sum) or multiply-add (GEMV) per element,
    the roofline is HBM-bound: every element read once."""
    import torch
    from tiled_staged_matmul_gb300 import binding, synthetic

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = synthetic.ROW_WORKLOADS[args.workload]
    X_h, x_h = w.operands()
    X = X_h.to(dev)
    x = x_h.to(dev) if x_h is not None else None
    out = torch.empty(w.R, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    working_set = w.algorithmic_bytes
    flush = working_set < 2 * L2_BYTES
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    sweep = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    sink = torch.empty(1, dtype=torch.float32, device=dev) if flush else None

    def flush_l2():
        scrub.zero_()
        torch.sum(sweep, dim=0, keepdim=True, out=sink)

    def call():
        if w.kind == "gemv":
            binding.check(binding.gemv_f16_f32acc(X.data_ptr(), x.data_ptr(), out.data_ptr(), w.R,
                                                  w.C, w.C, 1, stream.cuda_stream))
        else:
            binding.check(binding.rowsum_f32acc(X.data_ptr(), w.elem, out.data_ptr(), w.R, w.C, w.C,
                                                1, stream.cuda_stream))

    per_step_ms, t0, t1, sampler, burst_ms = timed_loop(args, call, flush_l2 if flush else None,
                                                        stream, world, local_rank)
    ms_local = sum(per_step_ms) / len(per_step_ms)
    clocks = sampler.summary(t0, t1)
    value, ms = replica_throughput(w.flops, ms_local, world, dev)
    roofline = roofline_of(w.flops, w.algorithmic_bytes, ms_local, recorded_traffic(w.name),
                           "tsm_row_reduce_kernel", clocks)
    result = {
        "metric": METRIC, "value": round(value, 4), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.elem, "data": "synthetic",
        "config": {"workload": w.name, "kind": w.kind, "R": w.R, "C": w.C, "elem": w.elem,
                   "seed": w.seed, "accumulate": "f32",
                   "l2": "flushed before every step (write 2xL2, then read 2xL2)" if flush else
                         f"inputs {working_set / 2**20:.0f} MiB > L2, no flush",
                   "parallelism": f"replicas x{world}"},
        "gpu_launches": args.steps,
        "roofline": roofline,
        "hbm_gbs": round(w.algorithmic_bytes / (ms_local * 1e-3) / 1e9, 1),
    }
    result["clocks"] = {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")}
    return result


def run_ours(args, rank, local_rank, world):
    import torch
    from tiled_staged_matmul_gb300 import binding, synthetic

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = pick_workload(args)
    A_h, B_h = synthetic.workload_operands(w)
    pad = args.ld_pad
    out_dtype = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[args.out]
    out_bytes = 4 if args.out == "f32" else 2
    lda, ldb, ldc = w.K + pad, w.N + pad, w.N + pad
    A = torch.empty((w.M, lda), dtype=torch.float16, device=dev)[:, :w.K]
    B = torch.empty((w.K, ldb), dtype=torch.float16, device=dev)[:, :w.N]
    A.copy_(A_h)
    B.copy_(B_h)
    C = torch.empty((w.M, ldc), dtype=out_dtype, device=dev)[:, :w.N]
    bias = (torch.linspace(-1, 1, w.N, dtype=torch.float32, device=dev) if args.bias else None)
    fused = args.act != "none" or args.bias or args.out != "f32"
    epi = binding.epilogue(1.0, bias.data_ptr() if bias is not None else 0, 0, args.act, 0.01,
                           args.out) if fused else None
    stream = torch.cuda.current_stream()
    opts = binding.GemmOptions(args.split_k, args.tile_n, 0, 0, args.tile_m, args.splitk_reduce)
    opts.red_cluster = args.red_cluster
    plan = binding.gemm_plan(w.M, w.N, w.K, 1, opts)
    launches_per_call = 2 if plan["split_k"] > 1 and not plan["fused_reduce"] else 1
    # Row pitches that are not multiples of 16 bytes: that operand is copied
    # (A and B in, C out) around the GEMM.
    copies = int(lda % 8 != 0) + int(ldb % 8 != 0) + int(ldc % (16 // out_bytes) != 0)
    repacked = copies > 0
    launches_per_call += copies

    working_set = 2 * w.M * w.K + 2 * w.K * w.N + out_bytes * w.M * w.N
    flush = working_set < 2 * L2_BYTES
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    sweep = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    sink = torch.empty(1, dtype=torch.float32, device=dev) if flush else None

    def flush_l2():
        # Write a buffer twice the L2, then read another one: the inputs are
        # evicted and the L2 is left holding clean lines, so the timed GEMM
        # does not pay for writing back the scrub's dirty lines.
        scrub.zero_()
        torch.sum(sweep, dim=0, keepdim=True, out=sink)

    def call(o=opts):
        if fused:
            binding.check(binding.gemm_f16_fused(A.data_ptr(), B.data_ptr(), C.data_ptr(), w.M, w.N,
                                                 w.K, lda, ldb, ldc, 0, 0, 0, 1, epi, o,
                                                 stream.cuda_stream))
        else:
            binding.check(binding.gemm_f16_f32acc_opts(A.data_ptr(), B.data_ptr(), C.data_ptr(),
                                                       w.M, w.N, w.K, lda, ldb, ldc, 0, 0, 0, 1,
                                                       o, stream.cuda_stream))

    per_step_ms, t0, t1, sampler, burst_ms = timed_loop(args, call, flush_l2 if flush else None,
                                                        stream, world, local_rank)
    ms_local = sum(per_step_ms) / len(per_step_ms)
    clocks = sampler.summary(t0, t1)
    value, ms = replica_throughput(w.flops, ms_local, world, dev)
    abytes = 2 * w.M * w.K + 2 * w.K * w.N + out_bytes * w.M * w.N + (4 * w.N if args.bias else 0)
    roofline = roofline_of(w.flops, abytes, ms_local,
                           recorded_traffic(w.name) if not pad and not fused else None,
                           "tsm_gemm_tcgen05_kernel" + (" + tsm_splitk_reduce_kernel"
                                                        if plan["split_k"] > 1
                                                        and not plan["fused_reduce"] else "")
                           + (f" + {copies} x tsm_repack_kernel" if repacked else ""), clocks)

    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K,
                   "dist": w.dist, "seed": w.seed, "accumulate": "f32",
                   "tile_m": plan["tile_m"], "tile_n": plan["tile_n"], "split_k": plan["split_k"],
                   "split_tail": (f"{plan['tail_tiles']} tiles of the last wave split "
                                  f"{plan['tail_split']} ways "
                                  + ("in column slices" if plan["tail_narrow"] else "along K")
                                  if plan["tail_split"] else "none"),
                   "red_cluster": plan["red_cluster"],
                   "splitk_sum": ("in-kernel" if plan["fused_reduce"] else "separate kernel")
                   if plan["split_k"] > 1 or (plan["tail_split"] and not plan["tail_narrow"])
                   else "none",
                   "stages": plan["stages"], "grid": plan["grid"],
                   "ld": [lda, ldb, ldc],
                   "epilogue": ({"activation": args.act, "bias": bool(args.bias), "out": args.out}
                                if fused else "none (f32 store)"),
                   "layout": (f"repacked ({copies} operand copies: row pitches not multiples "
                              "of 16 bytes)" if repacked else "TMA-addressable"),
                   "l2": "flushed before every step (write 2xL2, then read 2xL2)" if flush else
                         f"inputs+output {working_set / 2**20:.0f} MiB > L2, no flush",
                   "parallelism": f"replicas x{world}"},
        "gpu_launches": args.steps * launches_per_call,
        "roofline": roofline,
        "burst": burst_of(w.flops, abytes, burst_ms),
    }
    result["ms_per_step_stats"] = step_stats(per_step_ms)
    result["clocks"] = {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")}
    if args.trace:
        result["trace"] = traced_step(args, binding, call, plan, flush_l2 if flush else None, dev)
    plain_default = (args.workload == DEFAULT_WORKLOAD and not args.shape and not fused
                     and not pad and not (args.tile_m or args.tile_n or args.split_k
                                          or args.splitk_reduce or args.red_cluster))
    if plain_default and not args.no_workloads:
        # The other four shapes, interleaved, in the same run.
        table, _ = time_workloads(args, SIDE_WORKLOADS, dev, world, local_rank,
                                  max(args.workload_rounds, 10),
                                  headline=(w.name, per_step_ms, result["clocks"]))
        result["workloads"] = table
        result["binding_us_per_call"] = ctypes_us_per_call()
        result["gpu_launches"] += len(SIDE_WORKLOADS) * max(args.workload_rounds, 10)
        result["gpu_launches"] += sum(e["warm_l2"]["steps"] for e in table.values() if "warm_l2" in e)

    if not args.no_e2e and not fused:
        result["e2e"] = run_e2e(args, w, A_h, B_h, dev, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, A_h, B_h, target_s=15.0,
                                              C_gpu=C if plain_default else None)
    return result


# The other four GEMM shapes timed beside the headline in the same run
# (the small-integer twin of 64 x 128 x 128 is a parity case only).
SIDE_WORKLOADS = ("gemm_64x128x128_uniform", "gemm_1000x1000x1000_normal",
                  "gemm_4096x4096x4096_normal_invsqrtk", "gemm_256x256x65536_uniform")


def time_workloads(args, names, dev, world, local_rank, rounds: int, headline=None):
    """Time several GEMM workloads in one interleaved loop: every round runs
    one step of each (L2 flushed before each step whose inputs fit in it),
    each step bracketed by CUDA events on the launching stream, clocks
    sampled throughout.  Per workload: mean, median and minimum time per
    step, the roofline of the mean, median and best step, the in-kernel span
    of one traced step (first CTA entry to last CTA exit, %globaltimer: the
    kernel alone, without the launch) and the clocks of the loop.
    ``headline`` (name, per-step ms list, clocks) adds the headline
    workload's own timed steps to the table."""
    import torch
    from tiled_staged_matmul_gb300 import binding, synthetic

    stream = torch.cuda.current_stream()
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    sweep = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    sink = torch.empty(1, dtype=torch.float32, device=dev)

    def flush_l2():
        scrub.zero_()
        torch.sum(sweep, dim=0, keepdim=True, out=sink)

    runs = []
    for name in names:
        w = synthetic.WORKLOADS[name]
        A_h, B_h = synthetic.workload_operands(w)
        A, B = A_h.to(dev), B_h.to(dev)
        C = torch.empty((w.M, w.N), dtype=torch.float32, device=dev)
        working_set = 2 * w.M * w.K + 2 * w.K * w.N + 4 * w.M * w.N

        def call(w=w, A=A, B=B, C=C, o=None):
            if o is None:
                binding.check(binding.gemm_f16_f32acc(A.data_ptr(), B.data_ptr(), C.data_ptr(),
                                                      w.M, w.N, w.K, w.K, w.N, w.N,
                                                      stream.cuda_stream))
            else:
                binding.check(binding.gemm_f16_f32acc_opts(A.data_ptr(), B.data_ptr(),
                                                           C.data_ptr(), w.M, w.N, w.K, w.K, w.N,
                                                           w.N, 0, 0, 0, 1, o, stream.cuda_stream))
        runs.append((w, call, working_set < 2 * L2_BYTES, [], (A, B, C)))

    sampler = ClockSampler(local_rank)
    sampler.start()
    for _ in range(max(args.warmup, 3)):
        for w, call, flush, _, _ in runs:
            if flush:
                flush_l2()
            call()
    torch.cuda.synchronize()
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(rounds)] for _ in runs]
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    for r in range(rounds):
        for i, (w, call, flush, _, _) in enumerate(runs):
            if flush:
                flush_l2()
            ev[i][r][0].record(stream)
            call()
            ev[i][r][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    time.sleep(ClockSampler.LAG_S + 0.1)
    sampler.stop()
    binding.check(binding.gemm_get_device_status(stream.cuda_stream))
    clocks = sampler.summary(t0, t1)
    clocks = {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")}

    out = {}
    table = [(w, [e0.elapsed_time(e1) for e0, e1 in ev[i]], call, flush)
             for i, (w, call, flush, _, _) in enumerate(runs)]
    head_clocks = None
    if headline is not None:
        table.append((synthetic.WORKLOADS[headline[0]], headline[1], None, False))
        head_clocks = headline[2]
    for w, ms_list, call, flush in table:
        st = step_stats(ms_list)
        plan = binding.gemm_plan(w.M, w.N, w.K, 1, None)
        entry = {
            "M": w.M, "N": w.N, "K": w.K, "dist": w.dist, "seed": w.seed,
            "plan": {k: plan[k] for k in ("tile_m", "tile_n", "split_k", "fused_reduce",
                                          "red_cluster", "tail_split", "tail_narrow", "grid")},
            "steps": len(ms_list), "ms_per_step": st,
            "value": round(w.flops / (st["mean"] * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
            "l2": ("flushed before every step (write 2xL2, then read 2xL2)" if flush else
                   "inputs+output > L2, no flush"),
        }
        roof = roofline_of(w.flops, w.algorithmic_bytes, st["mean"],
                           recorded_traffic(w.name), "tsm_gemm_tcgen05_kernel",
                           clocks if call is not None else head_clocks)
        roof["frac_median"] = round(roof["frac"] * st["mean"] / st["median"], 4)
        roof["frac_best"] = round(roof["frac"] * st["mean"] / st["min"], 4)
        entry["roofline"] = roof
        entry["clocks"] = clocks if call is not None else head_clocks
        if call is not None and flush:
            entry["warm_l2"] = warm_l2_steps(call, w, stream, max(rounds // 2, 10))
        if call is not None:
            entry["host_us_per_call"] = host_us_per_call(call)
            span = kernel_span_us(binding, call, plan, flush_l2 if flush else None, dev)
            if span:
                entry["kernel_span_us"] = span
                entry["kernel_span_roofline_frac"] = round(
                    roof["frac"] * st["mean"] * 1e3 / span, 4)
        out[w.name] = entry
    return out, clocks


def warm_l2_steps(call, w, stream, steps: int) -> dict:
    """The same workload with no L2 flush between steps (its inputs stay
    L2-resident): back-to-back steps, each bracketed by CUDA events."""
    import torch
    for _ in range(3):
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for e0, e1 in ev:
        e0.record(stream)
        call()
        e1.record(stream)
    torch.cuda.synchronize()
    st = step_stats([e0.elapsed_time(e1) for e0, e1 in ev])
    return {"label": "warm L2: no flush between steps, inputs L2-resident", "steps": steps,
            "ms_per_step": st, "value": round(w.flops / (st["mean"] * 1e-3) / 1e12, 3),
            "unit": "TFLOP/s"}


def host_us_per_call(call, calls: int = 200) -> float:
    """Host time of one call through the C ABI (argument checks, planning,
    tensor maps, the launch), the GPU idle before each: median over
    ``calls`` calls, each timed on its own with the device synchronised
    outside the timing.  It includes the Python binding's ctypes call."""
    import torch
    times = []
    for _ in range(calls):
        torch.cuda.synchronize()
        t = time.perf_counter()
        call()
        times.append(time.perf_counter() - t)
    torch.cuda.synchronize()
    return round(statistics.median(times) * 1e6, 2)


def ctypes_us_per_call(calls: int = 2000) -> float:
    """The binding's own cost: median host time of a C ABI call that does
    nothing (gemm_version) through the same ctypes path."""
    from tiled_staged_matmul_gb300 import binding
    times = []
    for _ in range(calls):
        t = time.perf_counter()
        binding.gemm_version()
        times.append(time.perf_counter() - t)
    return round(statistics.median(times) * 1e6, 3)


def kernel_span_us(binding, call, plan, flush, dev, repeats: int = 5):
    """The GEMM kernel alone: first CTA entry to last CTA exit of one step,
    read from the kernel's own %globaltimer trace (median of a few flushed
    steps).  Launch latency and the events' own cost are outside it."""
    import torch
    spans = []
    for _ in range(repeats):
        tr = torch.zeros((plan["grid"], 8), dtype=torch.int64, device=dev)
        o = binding.GemmOptions(0, 0, 0, 0, 0, 0, 0, 0, tr.data_ptr())
        if flush:
            flush()
        call(o=o)
        torch.cuda.synchronize()
        t = tr.cpu()
        entry, exit_ = t[:, 0], t[:, 7]
        if (entry > 0).sum() == 0 or (exit_ > 0).sum() == 0:
            return None
        spans.append(float(exit_[exit_ > 0].max() - entry[entry > 0].min()) / 1000.0)
    return round(statistics.median(spans), 2)


TRACE_PHASES = ("entry", "setup", "first_data", "last_mma", "acc_ready", "stored", "reduced",
                "exit")


def traced_step(args, binding, call, plan, flush, dev):
    """One more step with the kernel's per-CTA trace on: for every phase, the
    min / median / max over CTAs of its time after the first CTA started
    (us; the timer ticks in steps of about 0.25 us)."""
    import torch
    tr = torch.zeros((plan["grid"], 8), dtype=torch.int64, device=dev)
    o = binding.GemmOptions(args.split_k, args.tile_n, 0, 0, args.tile_m, args.splitk_reduce,
                            0, 0, tr.data_ptr())
    o.red_cluster = args.red_cluster
    if flush:
        flush()
    call(o)
    torch.cuda.synchronize()
    t = tr.cpu().double()
    t0 = t[:, 0][t[:, 0] > 0].min()
    out = {}
    for i, name in enumerate(TRACE_PHASES):
        col = t[:, i][t[:, i] > 0]
        if col.numel():
            rel = ((col - t0) / 1000.0).sort().values
            out[name] = [round(float(rel[0]), 2), round(float(rel[rel.numel() // 2]), 2),
                         round(float(rel[-1]), 2)]
    return {"unit": "us after the first CTA entered, [min, median, max] over CTAs", **out}


def pick_workload(args):
    from tiled_staged_matmul_gb300 import synthetic
    if args.shape:
        M, N, K = (int(x) for x in args.shape.lower().split("x"))
        return synthetic.Workload(f"gemm_{M}x{N}x{K}_normal_invsqrtk", M, N, K,
                                  "normal_invsqrtk", 2000)
    return synthetic.WORKLOADS[args.workload]


def run_e2e(args, w, A_h, B_h, dev, world):
    """Same metric through the public API from pinned host buffers: every step
    copies that step's A and B to the device, runs the GEMM and copies its C
    back (``binding.HostPipeline``: three buffer sets, so the upload of one
    step overlaps the GEMM and download of the previous ones)."""
    import torch
    from tiled_staged_matmul_gb300 import binding

    depth = 3  # an upload waits only for the download three steps back
    A_p = A_h.pin_memory()
    B_p = B_h.pin_memory()
    C_p = [torch.empty((w.M, w.N), dtype=torch.float32).pin_memory() for _ in range(depth)]
    pipe = binding.HostPipeline(w.M, w.N, w.K, depth=depth, device=dev)
    for i in range(2 * depth):
        pipe.submit(A_p, B_p, C_p[i % depth])
    pipe.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(pipe.s_in)
    for i in range(args.e2e_steps):
        pipe.submit(A_p, B_p, C_p[i % depth])
    end.record(pipe.s_out)
    pipe.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    binding.check(binding.gemm_get_device_status(pipe.s_gemm.cuda_stream))
    ms = start.elapsed_time(end) / args.e2e_steps
    ms = max_over_ranks(ms, world, dev)
    return {"value": round(world * w.flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "pipeline_depth": depth, "steps": args.e2e_steps,
            "h2d_bytes_per_step": A_p.numel() * 2 + B_p.numel() * 2,
            "d2h_bytes_per_step": C_p[0].numel() * 4}


# ------------------------------------------------------------------ the oracle, timed

def oracle_sample_rows(w, A_h, B_h, rows: int, seed: int = 0, keep: bool = False):
    """Time the oracle on `rows` consecutive rows of C (a contiguous row
    panel of A times all of B): flops = 2 * rows * N * K.  With ``keep``,
    also return (first row, the fp64 rows)."""
    import oracle
    r0 = (seed * 7919) % max(1, w.M - rows + 1)
    A_rows = A_h[r0:r0 + rows].contiguous()
    t = time.perf_counter()
    ref = oracle.gemm_f64(A_rows, B_h, rows, w.N, w.K)
    dt = time.perf_counter() - t
    return (dt, r0, ref) if keep else dt


def cpu_baseline(w, A_h, B_h, target_s: float, C_gpu=None):
    """The oracle timed on a bounded row sample of the workload.  With
    ``C_gpu`` (the GPU's C of that workload) the rows it computed are also
    compared with the GPU's, at the tolerances the parity tests use."""
    import numpy as np
    import oracle
    probe_rows = max(1, min(w.M, int(2e9 // (2 * w.N * w.K)) or 1))
    dt = oracle_sample_rows(w, A_h, B_h, probe_rows)
    rate = 2 * probe_rows * w.N * w.K / max(dt, 1e-9)
    rows = max(1, min(w.M, int(rate * target_s / (2 * w.N * w.K))))
    dt, r0, ref = oracle_sample_rows(w, A_h, B_h, rows, seed=1, keep=True)
    flops = 2 * rows * w.N * w.K
    out = {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.threads(),
           "kind": "oracle", "seconds": round(dt, 2),
           "sample": f"{rows} of {w.M} rows of C ({rows} x {w.N} x {w.K}), fp64 triple loop, "
                     f"OpenMP over rows"}
    if C_gpu is not None:
        got = C_gpu[r0:r0 + rows].cpu().numpy().astype(np.float64)
        err = float(np.abs(got - ref).max())
        rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
        tol = 1e-3 * math.sqrt(w.K)
        out["parity"] = {"rows": [r0, r0 + rows], "max_abs_err": err, "rel_fro_err": rel,
                         "tol_max_abs": tol, "tol_rel_fro": 1e-4,
                         "finite": bool(np.isfinite(got).all()),
                         "pass": bool(err <= tol and rel <= 1e-4 and np.isfinite(got).all())}
    return out


def grouped_cpu_baseline(w, A_h, B_h, counts_h, target_s: float):
    """The oracle on a bounded sample of a grouped workload: the first rows
    of the busiest experts, in turn, until about ``target_s`` seconds."""
    import oracle
    order = sorted(range(w.groups), key=lambda g: -int(counts_h[g]))
    per_row = 2 * w.N * w.K
    t_total, flops, used = 0.0, 0, []
    rows = 1
    for g in order:
        r = min(int(counts_h[g]), rows)
        if r == 0:
            continue
        t = time.perf_counter()
        oracle.gemm_f64(A_h[g, :r].contiguous(), B_h[g], r, w.N, w.K)
        dt = time.perf_counter() - t
        t_total += dt
        flops += r * per_row
        used.append((g, r))
        if t_total >= target_s:
            break
        rows = max(1, min(w.M, int(r * (target_s - t_total) / max(dt, 1e-6) / 4)))
    return {"value": round(flops / max(t_total, 1e-9) / 1e12, 6), "unit": "TFLOP/s",
            "cores": oracle.threads(), "kind": "oracle", "seconds": round(t_total, 2),
            "sample": f"{sum(r for _, r in used)} routed rows from {len(used)} experts "
                      f"(x {w.N} x {w.K}), fp64 triple loop, OpenMP over rows"}


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, each step a bounded row sample."""
    import oracle
    from tiled_staged_matmul_gb300 import synthetic

    if args.workload in synthetic.GROUPED_WORKLOADS and not args.shape:
        return run_grouped_reference(args, world)
    w = pick_workload(args)
    A_h, B_h = synthetic.workload_operands(w)
    rows = max(1, min(w.M, int(4e9 // (2 * w.N * w.K)) or 1))
    for i in range(max(args.warmup, 0)):
        oracle_sample_rows(w, A_h, B_h, rows, seed=i)
    times = [oracle_sample_rows(w, A_h, B_h, rows, seed=i) for i in range(args.steps)]
    t = sum(times) / len(times)
    flops = 2 * rows * w.N * w.K
    value = flops / t / 1e12
    sample = f"{rows} of {w.M} rows of C per step ({rows} x {w.N} x {w.K}), fp64 triple loop"
    return {
        "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "dist": w.dist,
                   "seed": w.seed},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_grouped_reference(args, world):
    """The reference arm on a grouped workload: each step the oracle computes
    a bounded sample of routed rows (the first rows of the busiest expert)."""
    import oracle
    from tiled_staged_matmul_gb300 import synthetic

    w = synthetic.GROUPED_WORKLOADS[args.workload]
    A_h, B_h = synthetic.grouped_operands(w)
    counts = w.counts()
    g = int(max(range(w.groups), key=lambda e: int(counts[e])))
    rows = max(1, min(int(counts[g]), int(4e9 // (2 * w.N * w.K)) or 1))

    def step():
        t = time.perf_counter()
        oracle.gemm_f64(A_h[g, :rows].contiguous(), B_h[g], rows, w.N, w.K)
        return time.perf_counter() - t

    for _ in range(max(args.warmup, 0)):
        step()
    times = [step() for _ in range(args.steps)]
    t = sum(times) / len(times)
    value = 2 * rows * w.N * w.K / t / 1e12
    sample = (f"{rows} routed rows of expert {g} per step ({rows} x {w.N} x {w.K}), "
              "fp64 triple loop")
    return {
        "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": w.name, "groups": w.groups, "M": w.M, "N": w.N, "K": w.K,
                   "dist": w.dist, "seed": w.seed},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    from tiled_staged_matmul_gb300 import synthetic
    if args.workload in synthetic.GROUPED_WORKLOADS:
        result = run_grouped(args, rank, local_rank, world)
    elif args.workload in synthetic.ROW_WORKLOADS:
        result = run_rows(args, rank, local_rank, world)
    else:
        result = run_ours(args, rank, local_rank, world)
    if rank == 0:
        result["config"]["warm_up"] = (f"{max(args.warmup, 3)} steps, then steps until the GPU "
                                       f"had been busy {args.warm_seconds:g} s")
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

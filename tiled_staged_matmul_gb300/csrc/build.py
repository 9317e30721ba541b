"""Build ``libtsm_gemm.so`` in-tree with nvcc for sm_103a only.

The translation units compile in parallel: the plain GEMM kernels and the
cluster split-K sums, the fused-epilogue GEMM kernels once per activation
(``gemm_epi.cu`` with ``-DTSM_EPI_ACT``), the row-reduction kernels and the
host API.  The kernel units are compiled with ``-Xptxas -v`` and the build
fails if ptxas reports any spill stores or loads (only ptxas's printed
summary is read).
"""
from __future__ import annotations

import os
import re
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
PKG = os.path.dirname(HERE)
REPO = os.path.dirname(PKG)
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libtsm_gemm.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
PTXAS_LOG = os.path.join(BUILD_DIR, "ptxas.log")

# (source, object name, extra nvcc flags); the activations are gemm_internal.h's kAct* values
ACTIVATIONS = ["none", "relu", "leaky_relu", "gelu", "gelu_tanh", "silu"]
UNITS = ([("gemm_kernels.cu", "gemm_kernels", [])] +
         [("gemm_epi.cu", f"gemm_epi_{a}", [f"-DTSM_EPI_ACT={i}"]) for i, a in enumerate(ACTIVATIONS)] +
         [("rowsum_kernels.cu", "rowsum_kernels", []), ("gemm_api.cu", "gemm_api", [])])
SOURCES = sorted({u[0] for u in UNITS})
HEADERS = ["gemm_internal.h", "gemm_kernel.cuh", "ptx.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return cand


def _inputs() -> list[str]:
    files = [os.path.join(HERE, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(REPO, "include", "tsm_gemm.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _compile(src: str, obj: str, verbose_ptxas: bool, flags: list[str]) -> str:
    cmd = [_nvcc(), "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC", *flags,
           "-I", os.path.join(REPO, "include"), "-c", os.path.join(HERE, src), "-o", obj]
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def check_spills(log: str) -> None:
    bad = [ln for ln in log.splitlines()
           if re.search(r"(\d+) bytes spill (stores|loads)", ln)
           and not re.search(r"\b0 bytes spill stores, 0 bytes spill loads", ln)]
    if bad:
        raise RuntimeError("ptxas reports register spills:\n" + "\n".join(bad))


def build(force: bool = False, quiet: bool = True) -> str:
    if not force and up_to_date():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    objs = [os.path.join(BUILD_DIR, name + ".o") for _, name, _ in UNITS]
    kernel_unit = [src != "gemm_api.cu" for src, _, _ in UNITS]
    with ThreadPoolExecutor(len(UNITS)) as ex:
        logs = list(ex.map(lambda a: _compile(*a),
                           [(src, o, k, fl) for (src, _, fl), o, k in zip(UNITS, objs, kernel_unit)]))
    ptxas = "".join(log for log, k in zip(logs, kernel_unit) if k)
    with open(PTXAS_LOG, "w") as f:
        f.write(ptxas)
    check_spills(ptxas)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    r = subprocess.run([_nvcc(), *ARCH, "-shared", "-o", tmp, *objs],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    if not quiet:
        print(logs[0], file=sys.stderr)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, quiet=False))

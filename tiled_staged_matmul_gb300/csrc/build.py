"""Build ``libtsm_gemm.so`` in-tree with nvcc for sm_103a only.

Three translation units (the GEMM kernels, the row-reduction kernels, the
host API) compile in parallel; the kernel units are compiled with ``-Xptxas -v`` and the build fails if ptxas reports any
spill stores or loads (only ptxas's printed summary is read).
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

SOURCES = ["gemm_kernels.cu", "rowsum_kernels.cu", "gemm_api.cu"]
HEADERS = ["gemm_internal.h", "ptx.cuh"]
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


def _compile(src: str, obj: str, verbose_ptxas: bool) -> str:
    cmd = [_nvcc(), "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
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
    objs = [os.path.join(BUILD_DIR, os.path.splitext(s)[0] + ".o") for s in SOURCES]
    with ThreadPoolExecutor(len(SOURCES)) as ex:
        logs = list(ex.map(lambda a: _compile(*a),
                           [(s, o, s.endswith("_kernels.cu")) for s, o in zip(SOURCES, objs)]))
    with open(PTXAS_LOG, "w") as f:
        f.write(logs[0] + logs[1])
    check_spills(logs[0] + logs[1])
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

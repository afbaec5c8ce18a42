"""Build the CUDA library in-tree: ``csrc/*.cu`` -> ``libdtgemm.so`` for sm_103a.

nvcc cross-compiles without a GPU; the same command builds on the x86 host and on
the Arm GPU host.  The CUDA runtime is linked statically, so the library loads
without extra library paths.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libdtgemm.so")
# One translation unit for the host side, one per operand type for the kernels: they
# compile in parallel and link into one library.
SOURCES = [os.path.join(CSRC, f) for f in ("gemm_api.cu", "kernels_f16.cu", "kernels_bf16.cu", "kernels_e4m3.cu",
                                           "kernels_e5m2.cu", "kernels_mx.cu", "kernels_sparse.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in ("gemm_kernel.cuh", "sm103_ptx.cuh", "kernel_set.cuh")] + [
    os.path.join(INCLUDE, "gemm.h")]
OBJ_DIR = os.path.join(HERE, "_build")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = os.path.join(cand, "bin", "nvcc") if cand else ""
        if p and os.path.exists(p):
            return p
    p = shutil.which("nvcc")
    if not p:
        raise RuntimeError("nvcc not found: set CUDA_HOME")
    return p


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in DEPENDS)


def _run(cmd):
    return subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    nvcc = nvcc_path()
    os.makedirs(OBJ_DIR, exist_ok=True)
    common = [nvcc, *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    if verbose:
        common.insert(1, "-Xptxas=-v")
    jobs = []
    for src in SOURCES:
        obj = os.path.join(OBJ_DIR, os.path.splitext(os.path.basename(src))[0] + ".o")
        cmd = [*common, "-c", "-o", obj, src]
        jobs.append((cmd, obj, _run(cmd)))
    objs, logs, failed = [], [], None
    for cmd, obj, proc in jobs:
        out, _ = proc.communicate()
        logs.append(out)
        if proc.returncode != 0 and failed is None:
            failed = (cmd, proc.returncode, out)
        objs.append(obj)
    if failed:
        cmd, rc, out = failed
        raise RuntimeError(f"nvcc failed ({rc}):\n{' '.join(cmd)}\n{out}")
    link = [nvcc, *ARCH_FLAGS, "-shared", "-Xcompiler", "-fPIC", "-o", LIB + ".tmp", *objs]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed ({r.returncode}):\n{' '.join(link)}\n{r.stdout}\n{r.stderr}")
    if verbose:
        sys.stderr.write("".join(logs) + r.stdout + r.stderr)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)

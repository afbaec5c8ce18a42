"""The C ABI from a C program: tests/c_abi/gemm_c_consumer.c, built with gcc against
include/gemm.h and libdtgemm.so only (no Python, torch or CUDA headers in the program).

On the CPU it checks the host-side entry points; on a GB300 it also runs GEMMs on host
buffers through gemm_run_host in every configuration and compares them bit for bit with
the CPU oracle linked into the same program.
"""
import ctypes
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "gemm_c_consumer.c")
ORACLE_C = os.path.join(ROOT, "oracle", "gemm_oracle.c")


def _build(tmp_path) -> str:
    from dense_tiled_gemm_04_gb300 import build

    lib = build.build()
    libdir = os.path.dirname(lib)
    exe = str(tmp_path / "gemm_c_consumer")
    cmd = ["gcc", "-std=c11", "-O1", "-ffp-contract=off", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           SRC, ORACLE_C, "-o", exe, "-L", libdir, "-ldtgemm", f"-Wl,-rpath,{libdir}", "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_program_host_entry_points(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe, "host"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "gemm_c_consumer host: ok" in r.stdout
    # The ctypes binding lays the ABI's structs out as the C compiler does.
    from dense_tiled_gemm_04_gb300 import native

    sizes = dict(zip(["gemm_plan_t", "gemm_args_t"], (int(x) for x in r.stdout.split("sizeof ")[1].split()[1::2])))
    assert sizes == {"gemm_plan_t": ctypes.sizeof(native.gemm_plan_t), "gemm_args_t": ctypes.sizeof(native.gemm_args_t)}


@pytest.mark.gpu
def test_c_program_gemm_run_host_bit_exact(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe, "gpu"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "gemm_c_consumer gpu: ok" in r.stdout

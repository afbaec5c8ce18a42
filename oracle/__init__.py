"""CPU oracle for the tiled dense contraction C = A·B.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The GPU
library never calls it and shares no code with it.

Two formulations live here:

* :func:`gemm` / :func:`gemm_rows` / :func:`gemm_elems` -- the plain definition
  ``C[m,n] = rne(sum_k A[m,k] * Beff[k,n])`` with an fp64 sum, in C
  (``gemm_oracle.c``), OpenMP over rows.
* :mod:`oracle.tiled` -- the pages' tile decomposition written out step by step
  (output tile grid, K-block loop, zero-filled tails, masked write-back), used to
  pin the direct definition against the worked example.

Inputs are 16-bit codes: numpy ``uint16`` arrays (or torch CPU tensors of dtype
float16/bfloat16, whose bit patterns are taken as they are).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_gemm.so")

LAYOUTS = {"NN": 0, "TN": 1}
DTYPES = {"f16": 0, "bf16": 1, "e4m3": 2, "e5m2": 3}

_lib = None


def build(force: bool = False) -> str:
    """Compile ``gemm_oracle.c`` into ``liboracle_gemm.so`` (gcc, OpenMP if available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", _LIB + ".tmp", _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    i64, p = ctypes.c_int64, ctypes.c_void_p
    lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_f64.restype = ctypes.c_double
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f64.restype = ctypes.c_double
    lib.oracle_f64_to_f16.argtypes = [ctypes.c_double]
    lib.oracle_f64_to_f16.restype = ctypes.c_uint16
    lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
    lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
    lib.oracle_gemm_rows.argtypes = [p, p, i64, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                     p, i64, p, p, i64, ctypes.c_int]
    lib.oracle_gemm_rows.restype = ctypes.c_int
    lib.oracle_gemm_elems.argtypes = [p, p, i64, i64, i64, ctypes.c_int, ctypes.c_int, p, p, i64, p, p]
    lib.oracle_gemm_elems.restype = ctypes.c_int
    lib.oracle_gemm_rows_axpby.argtypes = [p, p, p, i64, i64, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_double, ctypes.c_double, p, i64, p, p, i64, ctypes.c_int]
    lib.oracle_gemm_rows_axpby.restype = ctypes.c_int
    lib.oracle_gemm_rows_typed.argtypes = [p, p, p, i64, i64, i64, i64, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_double, ctypes.c_double, p, i64, p, p, i64, ctypes.c_int]
    lib.oracle_gemm_rows_typed.restype = ctypes.c_int
    lib.oracle_gemm_rows_blockscaled.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64, i64, i64, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double, p, i64,
                                                 p, p, i64, ctypes.c_int]
    lib.oracle_gemm_rows_blockscaled.restype = ctypes.c_int
    lib.oracle_sparse24_compress.argtypes = [p, i64, i64, i64, p, i64, p, i64]
    lib.oracle_sparse24_compress.restype = i64
    lib.oracle_gemm_rows_sparse24.argtypes = [p, p, p, p, i64, i64, i64, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_double, ctypes.c_double, p, i64, p, p, i64, ctypes.c_int]
    lib.oracle_gemm_rows_sparse24.restype = ctypes.c_int
    lib.oracle_e8m0_to_f64.argtypes = [ctypes.c_uint8]
    lib.oracle_e8m0_to_f64.restype = ctypes.c_double
    lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_f64.restype = ctypes.c_double
    lib.oracle_e5m2_to_f64.argtypes = [ctypes.c_uint8]
    lib.oracle_e5m2_to_f64.restype = ctypes.c_double
    lib.oracle_decode_array.argtypes = [p, p, i64, ctypes.c_int]
    lib.oracle_decode_array.restype = None
    lib.oracle_encode_array.argtypes = [p, p, i64, ctypes.c_int]
    lib.oracle_encode_array.restype = None
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    _lib = lib
    return lib


def _codes(x) -> np.ndarray:
    """16-bit codes of x as a numpy uint16 array (a view where possible)."""
    if isinstance(x, np.ndarray):
        if x.dtype == np.uint16:
            return x
        if x.dtype == np.float16:
            return x.view(np.uint16)
        raise TypeError(f"unsupported numpy dtype {x.dtype}")
    import torch  # torch CPU tensors only: bit patterns are taken unchanged

    if x.dtype in (torch.float8_e4m3fn, torch.float8_e5m2, torch.uint8):
        # 8-bit codes widened to 16 bits (the C side reads the low byte)
        return x.detach().cpu().view(torch.uint8).numpy().astype(np.uint16)
    if x.dtype not in (torch.float16, torch.bfloat16, torch.int16):
        raise TypeError(f"unsupported torch dtype {x.dtype}")
    return x.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def _ld(x: np.ndarray) -> int:
    """Leading dimension (elements) of a 2-D row-major array with unit column stride."""
    if x.ndim != 2:
        raise ValueError("expected a 2-D array")
    if x.size == 0 or x.shape[0] <= 1:
        return max(x.shape[1], 1)
    if x.strides[1] != 2 and x.shape[1] > 1:
        raise ValueError("expected unit column stride")
    if x.shape[1] == 0:
        return max(x.shape[1], 1)
    return x.strides[0] // 2


def decode(codes, dtype: str) -> np.ndarray:
    """Exact fp64 values of 16-bit codes (through the C decoder)."""
    lib = _load()
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint16))
    out = np.empty(c.shape, dtype=np.float64)
    lib.oracle_decode_array(c.ctypes.data, out.ctypes.data, c.size, DTYPES[dtype])
    return out


def encode(values, dtype: str) -> np.ndarray:
    """Round fp64 values to 16-bit codes, nearest-even (through the C encoder)."""
    lib = _load()
    v = np.ascontiguousarray(np.asarray(values, dtype=np.float64))
    out = np.empty(v.shape, dtype=np.uint16)
    lib.oracle_encode_array(v.ctypes.data, out.ctypes.data, v.size, DTYPES[dtype])
    return out


def _shape_check(A: np.ndarray, B: np.ndarray, layout: str):
    M, K = A.shape
    if layout == "NN":
        Kb, N = B.shape
    elif layout == "TN":
        N, Kb = B.shape
    else:
        raise ValueError(layout)
    if Kb != K:
        raise ValueError(f"K mismatch: A is {A.shape}, B is {B.shape} ({layout})")
    return M, N, K


def gemm_rows(A, B, layout: str, dtype: str, rows, want_f64: bool = False, nthreads: int = 0):
    """Rows ``rows`` of C (rounded codes, shape (len(rows), N)); plus the fp64 sums if asked.

    Returns ``(codes, f64_or_None, threads_used)``.
    """
    lib = _load()
    A, B = _codes(A), _codes(B)
    M, N, K = _shape_check(A, B, layout)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if rows.size and (rows.min() < 0 or rows.max() >= M):
        raise IndexError("row out of range")
    out16 = np.zeros((rows.size, N), dtype=np.uint16)
    out64 = np.zeros((rows.size, N), dtype=np.float64) if want_f64 else None
    lda, ldb = _ld(A), _ld(B)
    used = lib.oracle_gemm_rows(
        A.ctypes.data, B.ctypes.data, N, K, lda, ldb, LAYOUTS[layout], DTYPES[dtype],
        rows.ctypes.data, rows.size, out16.ctypes.data,
        out64.ctypes.data if out64 is not None else None, N, int(nthreads))
    if used < 0:
        raise MemoryError("oracle allocation failed")
    return out16, out64, used


def gemm(A, B, layout: str, dtype: str, want_f64: bool = False, nthreads: int = 0):
    """All of C: rounded codes (M, N) uint16, or ``(codes, f64)`` if ``want_f64``."""
    A = _codes(A)
    codes, f64, _ = gemm_rows(A, B, layout, dtype, np.arange(A.shape[0]), want_f64, nthreads)
    return (codes, f64) if want_f64 else codes


def gemm_elems(A, B, layout: str, dtype: str, ms, ns, want_f64: bool = False):
    """Individual elements C[ms[i], ns[i]] (rounded codes; plus fp64 sums if asked)."""
    lib = _load()
    A, B = _codes(A), _codes(B)
    M, N, K = _shape_check(A, B, layout)
    ms = np.ascontiguousarray(np.asarray(ms, dtype=np.int64))
    ns = np.ascontiguousarray(np.asarray(ns, dtype=np.int64))
    if ms.shape != ns.shape:
        raise ValueError("ms and ns differ in shape")
    if ms.size and (ms.min() < 0 or ms.max() >= M or ns.min() < 0 or ns.max() >= N):
        raise IndexError("element out of range")
    out16 = np.zeros(ms.shape, dtype=np.uint16)
    out64 = np.zeros(ms.shape, dtype=np.float64) if want_f64 else None
    rc = lib.oracle_gemm_elems(A.ctypes.data, B.ctypes.data, K, _ld(A), _ld(B), LAYOUTS[layout],
                               DTYPES[dtype], ms.ctypes.data, ns.ctypes.data, ms.size,
                               out16.ctypes.data, out64.ctypes.data if out64 is not None else None)
    if rc != 0:
        raise MemoryError("oracle allocation failed")
    return (out16, out64) if want_f64 else out16


def gemm_axpby(A, B, layout: str, dtype: str, alpha: float, beta: float, Cin=None, rows=None,
               want_f64: bool = False, nthreads: int = 0):
    """alpha * (A·B) + beta * Cin (Cin: the logical M x N input codes, row-major; ignored when
    beta == 0).  Returns rounded codes for `rows` (default all), or ``(codes, f64)``."""
    lib = _load()
    A, B = _codes(A), _codes(B)
    M, N, K = _shape_check(A, B, layout)
    rows = np.arange(M) if rows is None else np.asarray(rows)
    rows = np.ascontiguousarray(rows.astype(np.int64))
    if beta != 0.0:
        Cin = np.ascontiguousarray(_codes(Cin))
        if Cin.shape != (M, N):
            raise ValueError(f"Cin must be {M} x {N}")
        cptr, ldcin = Cin.ctypes.data, max(N, 1)
    else:
        cptr, ldcin = None, 1
    out16 = np.zeros((rows.size, N), dtype=np.uint16)
    out64 = np.zeros((rows.size, N), dtype=np.float64) if want_f64 else None
    used = lib.oracle_gemm_rows_axpby(A.ctypes.data, B.ctypes.data, cptr, N, K, _ld(A), _ld(B), ldcin,
                                      LAYOUTS[layout], DTYPES[dtype], float(alpha), float(beta), rows.ctypes.data,
                                      rows.size, out16.ctypes.data,
                                      out64.ctypes.data if out64 is not None else None, N, int(nthreads))
    if used < 0:
        raise MemoryError("oracle allocation failed")
    return (out16, out64) if want_f64 else out16


def gemm_typed(A, B, layout: str, in_dtype: str, out_dtype: str, alpha: float = 1.0, beta: float = 0.0, Cin=None,
               rows=None, want_f64: bool = False, nthreads: int = 0):
    """alpha * (A·B) + beta * Cin with inputs of type ``in_dtype`` (f16, bf16, e4m3, e5m2) and
    the result / Cin of type ``out_dtype`` (f16, bf16).  Rounded codes for ``rows`` (default
    all), or ``(codes, f64)``."""
    lib = _load()
    A, B = _codes(A), _codes(B)
    M, N, K = _shape_check(A, B, layout)
    A, B = np.ascontiguousarray(A), np.ascontiguousarray(B)
    rows = np.arange(M) if rows is None else np.asarray(rows)
    rows = np.ascontiguousarray(rows.astype(np.int64))
    if beta != 0.0:
        Cin = np.ascontiguousarray(_codes(Cin))
        if Cin.shape != (M, N):
            raise ValueError(f"Cin must be {M} x {N}")
        cptr, ldcin = Cin.ctypes.data, max(N, 1)
    else:
        cptr, ldcin = None, 1
    out16 = np.zeros((rows.size, N), dtype=np.uint16)
    out64 = np.zeros((rows.size, N), dtype=np.float64) if want_f64 else None
    used = lib.oracle_gemm_rows_typed(A.ctypes.data, B.ctypes.data, cptr, N, K, _ld(A), _ld(B), ldcin,
                                      LAYOUTS[layout], DTYPES[in_dtype], DTYPES[out_dtype], float(alpha), float(beta),
                                      rows.ctypes.data, rows.size, out16.ctypes.data,
                                      out64.ctypes.data if out64 is not None else None, N, int(nthreads))
    if used < 0:
        raise MemoryError("oracle allocation failed")
    return (out16, out64) if want_f64 else out16


def _scales(x, rows: int, nblocks: int, what: str) -> np.ndarray:
    """Row-major uint8 exponent array of shape (rows, nblocks) (numpy or torch CPU)."""
    if not isinstance(x, np.ndarray):
        x = x.detach().cpu().numpy()
    x = np.ascontiguousarray(x, dtype=np.uint8)
    if x.shape != (rows, nblocks):
        raise ValueError(f"{what} must be {rows} x {nblocks}, got {x.shape}")
    return x


def gemm_blockscaled(A, B, sa, sb, layout: str, in_dtype: str, out_dtype: str, alpha: float = 1.0,
                     beta: float = 0.0, Cin=None, rows=None, want_f64: bool = False, nthreads: int = 0):
    """alpha * sum_j 2^(sa-127) 2^(sb-127) (A·B over K block j) + beta * Cin: 8-bit operands with
    one E8M0 scale per 32 K elements of each row of A (``sa``: M x ceil(K/32)) and of each
    column of Beff (``sb``: N x ceil(K/32)).  Rounded codes for ``rows``, or ``(codes, f64)``."""
    lib = _load()
    A, B = _codes(A), _codes(B)
    M, N, K = _shape_check(A, B, layout)
    A, B = np.ascontiguousarray(A), np.ascontiguousarray(B)
    nb = -(-K // 32)
    sa = _scales(sa, M, nb, "sa")
    sb = _scales(sb, N, nb, "sb")
    rows = np.arange(M) if rows is None else np.asarray(rows)
    rows = np.ascontiguousarray(rows.astype(np.int64))
    if beta != 0.0:
        Cin = np.ascontiguousarray(_codes(Cin))
        if Cin.shape != (M, N):
            raise ValueError(f"Cin must be {M} x {N}")
        cptr, ldcin = Cin.ctypes.data, max(N, 1)
    else:
        cptr, ldcin = None, 1
    out16 = np.zeros((rows.size, N), dtype=np.uint16)
    out64 = np.zeros((rows.size, N), dtype=np.float64) if want_f64 else None
    used = lib.oracle_gemm_rows_blockscaled(A.ctypes.data, B.ctypes.data, sa.ctypes.data, sb.ctypes.data, cptr, N, K,
                                            _ld(A), _ld(B), max(nb, 1), max(nb, 1), ldcin, LAYOUTS[layout],
                                            DTYPES[in_dtype], DTYPES[out_dtype], float(alpha), float(beta),
                                            rows.ctypes.data, rows.size, out16.ctypes.data,
                                            out64.ctypes.data if out64 is not None else None, N, int(nthreads))
    if used < 0:
        raise MemoryError("oracle allocation failed")
    return (out16, out64) if want_f64 else out16


def sparse24_compress(A):
    """2:4 compression of a dense 16-bit A (M x K, K % 4 == 0): (Ac codes M x K/2, metadata
    words M x ceil(K/32) uint32, number of groups with more than two non-zeros)."""
    lib = _load()
    A = np.ascontiguousarray(_codes(A))
    M, K = A.shape
    if K % 4:
        raise ValueError("K must be a multiple of 4")
    Ac = np.zeros((M, K // 2), dtype=np.uint16)
    lde = max(-(-K // 32), 1)
    E = np.zeros((M, lde), dtype=np.uint32)
    bad = lib.oracle_sparse24_compress(A.ctypes.data, M, K, max(K, 1), Ac.ctypes.data, max(K // 2, 1), E.ctypes.data,
                                       lde)
    return Ac, E[:, :-(-K // 32)] if K else E[:, :0], int(bad)


def gemm_sparse24(Ac, E, B, layout: str, dtype: str, alpha: float = 1.0, beta: float = 0.0, Cin=None, rows=None,
                  want_f64: bool = False, nthreads: int = 0):
    """alpha * (the sparse contraction of Ac, E with B) + beta * Cin; K = 2 * Ac's columns."""
    lib = _load()
    Ac = np.ascontiguousarray(_codes(Ac))
    B = np.ascontiguousarray(_codes(B))
    M, Kc = Ac.shape
    K = 2 * Kc
    N = B.shape[1] if layout == "NN" else B.shape[0]
    if (B.shape[0] if layout == "NN" else B.shape[1]) != K:
        raise ValueError(f"K mismatch: Ac is {Ac.shape} (K = {K}), B is {B.shape} ({layout})")
    E = np.ascontiguousarray(np.asarray(E, dtype=np.uint32))
    if E.shape != (M, -(-K // 32)):
        raise ValueError(f"E must be {M} x {-(-K // 32)}")
    rows = np.arange(M) if rows is None else np.asarray(rows)
    rows = np.ascontiguousarray(rows.astype(np.int64))
    if beta != 0.0:
        Cin = np.ascontiguousarray(_codes(Cin))
        cptr, ldcin = Cin.ctypes.data, max(N, 1)
    else:
        cptr, ldcin = None, 1
    out16 = np.zeros((rows.size, N), dtype=np.uint16)
    out64 = np.zeros((rows.size, N), dtype=np.float64) if want_f64 else None
    used = lib.oracle_gemm_rows_sparse24(Ac.ctypes.data, E.ctypes.data, B.ctypes.data, cptr, N, K, max(Kc, 1),
                                         max(E.shape[1], 1), _ld(B), ldcin, LAYOUTS[layout], DTYPES[dtype],
                                         float(alpha), float(beta), rows.ctypes.data, rows.size, out16.ctypes.data,
                                         out64.ctypes.data if out64 is not None else None, N, int(nthreads))
    if used < 0:
        raise MemoryError("oracle allocation failed")
    return (out16, out64) if want_f64 else out16


def e8m0(e: int) -> float:
    return float(_load().oracle_e8m0_to_f64(int(e)))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


__all__ = ["build", "decode", "encode", "gemm", "gemm_rows", "gemm_elems", "gemm_axpby", "gemm_typed",
           "gemm_blockscaled", "e8m0", "sparse24_compress", "gemm_sparse24", "max_threads",
           "LAYOUTS", "DTYPES"]

"""The pages' tile decomposition of C = A·B, written out step by step (fp64, numpy).

TEST INFRASTRUCTURE (part of the oracle): it pins the direct definition in
``gemm_oracle.c`` against the worked example of "NineToothed GEMM 语法入门"
(NineToothed GEMM syntax primer).  Small sizes only.

Steps, in the page's order and notation:

* §1 "print every level of the nested tensor": A (M, K) is cut into (BM, BK) tiles,
  the tile grid is grouped one tile-row at a time, expanded across the N tiles of the
  output and the singleton group axis squeezed away; B (K, N) likewise with (BK, BN)
  tiles grouped one tile-column at a time.  :func:`arrangement_shapes` reports the
  shape of every level.
* §2: one program per output tile; ``accumulator = zeros(BM, BN)``; for each K block
  ``accumulator += dot(lhs[k], rhs[k])``; ``output = accumulator``.
* §3: ``lhs[p][r, t] = A[i*BM + r, p*BK + t]``, ``rhs[p][t, s] = B[p*BK + t, j*BN + s]``,
  ``output[r, s] = C[i*BM + r, j*BN + s]``.
* §4: tile counts are ceil(M/BM), ceil(N/BN), ceil(K/BK).
* §5: a read outside M/N/K yields 0; a write outside M x N is dropped.

``numpy.matmul`` on one (BM, BK) x (BK, BN) block pair is the library step for ``dot``.
"""
from __future__ import annotations

import numpy as np


def cdiv(a: int, b: int) -> int:
    """ceil(a / b) for a >= 0, b > 0 (§4)."""
    return -(-a // b)


def grid(M: int, N: int, K: int, BM: int, BN: int, BK: int):
    """(M tiles, N tiles, K blocks), §4."""
    return cdiv(M, BM), cdiv(N, BN), cdiv(K, BK)


def arrangement_shapes(M: int, N: int, K: int, BM: int, BN: int, BK: int) -> dict:
    """Shape of every level of the nested A / B / C views after each step of §1.

    Each value is a list of tuples, outermost level first.
    """
    TM, TN, KB = grid(M, N, K, BM, BN, BK)
    return {
        "A original": [(M, K)],
        "A tiled": [(TM, KB), (BM, BK)],
        "A grouped": [(TM, 1), (1, KB), (BM, BK)],
        "A expanded": [(TM, TN), (1, KB), (BM, BK)],
        "A squeezed": [(TM, TN), (KB,), (BM, BK)],
        "B final": [(TM, TN), (KB,), (BK, BN)],
        "C final": [(TM, TN), (BM, BN)],
    }


def lhs_block(A: np.ndarray, i: int, p: int, BM: int, BK: int) -> np.ndarray:
    """lhs[p] of program (i, .): A[i*BM + r, p*BK + t], zero where outside A (§3, §5)."""
    M, K = A.shape
    blk = np.zeros((BM, BK), dtype=np.float64)
    for r in range(BM):
        for t in range(BK):
            if i * BM + r < M and p * BK + t < K:
                blk[r, t] = A[i * BM + r, p * BK + t]
    return blk


def rhs_block(B: np.ndarray, j: int, p: int, BK: int, BN: int) -> np.ndarray:
    """rhs[p] of program (., j): B[p*BK + t, j*BN + s], zero where outside B (§3, §5)."""
    K, N = B.shape
    blk = np.zeros((BK, BN), dtype=np.float64)
    for t in range(BK):
        for s in range(BN):
            if p * BK + t < K and j * BN + s < N:
                blk[t, s] = B[p * BK + t, j * BN + s]
    return blk


def tiled_gemm(A: np.ndarray, B: np.ndarray, BM: int, BN: int, BK: int, drop_last_k_block: bool = False):
    """C = A·B (fp64) computed one output tile at a time (§2-§5).

    ``A`` is (M, K) and ``B`` is (K, N), both as fp64 values (B is the logical K x N
    operand; a stored N x K array is passed transposed).  ``drop_last_k_block`` runs
    the K loop one block short: the mistake §8 exercise three is built to catch, kept
    here so a test can show the pin notices it.
    """
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    M, K = A.shape
    Kb, N = B.shape
    assert K == Kb
    TM, TN, KB = grid(M, N, K, BM, BN, BK)
    C = np.full((M, N), np.nan)
    k_blocks = KB - 1 if drop_last_k_block else KB
    for i in range(TM):
        for j in range(TN):
            acc = np.zeros((BM, BN), dtype=np.float64)          # accumulator = zeros
            for p in range(k_blocks):                             # for k in range(lhs.shape[0])
                acc += lhs_block(A, i, p, BM, BK) @ rhs_block(B, j, p, BK, BN)
            for r in range(BM):                                   # output = accumulator, masked
                for s in range(BN):
                    if i * BM + r < M and j * BN + s < N:
                        C[i * BM + r, j * BN + s] = acc[r, s]
    return C


def tail_valid_counts(M: int, N: int, K: int, BM: int, BN: int, BK: int):
    """Valid rows/cols of the bottom-right output tile and valid K of the last K block (§5)."""
    TM, TN, KB = grid(M, N, K, BM, BN, BK)
    return M - (TM - 1) * BM, N - (TN - 1) * BN, K - (KB - 1) * BK

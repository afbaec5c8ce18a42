"""Seeded synthetic inputs for the GEMM workloads.

This module holds the workload table and the random draws only -- no GEMM
arithmetic -- so that both the GPU path's tests/benchmark and the CPU oracle can
take their inputs from it.

Recipe: a CPU ``torch.Generator`` seeded with the workload's seed draws A (M x K)
first, then B in its *stored* shape (K x N for NN, N x K for TN), in fp32; the
values are scaled and rounded to the operand type (fp16, bf16, E4M3 or E5M2) by torch's
round-to-nearest-even cast.  Block scales (E8M0 exponents, one per 32 K elements of each
row of A and column of B) are drawn by a numpy generator seeded with seed + 1000,
uniform in {124..130} (scales 1/8 .. 8).  A sparse workload's A is pruned to a 2:4 pattern
along K (prune_24: two of the four positions of every group drawn uniformly from the six
pairs by a numpy generator seeded with seed + 2000).
Distributions: ``uniform`` = U[-1, 1) (``rand*2-1``), ``normal`` = N(0, 1)
(``randn``), ``int`` = integers uniform in {-2..2} (``randint(-2, 3)``).
A leading dimension larger than the row length pads each row with NaN, so a
kernel that reads past the logical edge poisons its own result.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    layout: str      # "NN": B stored K x N; "TN": B stored N x K
    dtype: str       # operand type: "f16" | "bf16" | "e4m3" | "e5m2"
    dist: str        # "uniform" | "normal" | "int" | "ones"
    scale: float     # multiplies the draw (1/sqrt(K) for the normalised workloads)
    seed: int
    out: str = ""    # type of C ("" = dtype; 8-bit operands: "f16" | "bf16")
    scales: str = "none"  # 8-bit operands: "tensor" (scale_a = scale_b = K^-1/4) | "block" (E8M0 per 32 K)
    sparse: bool = False  # A pruned to a 2:4 pattern along K (prune_24, seed + 2000)

    @property
    def out_dtype(self) -> str:
        return self.out or self.dtype

    @property
    def elem_bytes(self) -> int:
        return 1 if self.dtype in ("e4m3", "e5m2") else 2

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def algorithmic_bytes(self) -> int:
        """Read A and B (and their block scales) once, write the 16-bit C once.  A 2:4 A
        counts its kept half and 4 bits of positions per group of four."""
        sf = (self.M + self.N) * -(-self.K // 32) if self.scales == "block" else 0
        a = self.elem_bytes * self.M * self.K // 2 + self.M * self.K // 8 if self.sparse else \
            self.elem_bytes * self.M * self.K
        return a + self.elem_bytes * self.K * self.N + 2 * self.M * self.N + sf

    def with_dist(self, dist: str, scale: float = 1.0) -> "Workload":
        return replace(self, dist=dist, scale=scale)


WORKLOADS = {
    "c1": Workload("fp16 NN 128x256x192 (the page's worked example)", 128, 256, 192, "NN", "f16", "uniform", 1.0, 0),
    "c2": Workload("ragged fp16 TN 1000^3", 1000, 1000, 1000, "TN", "f16", "normal", 1.0, 1),
    "c3": Workload("square fp16 NN 4096^3", 4096, 4096, 4096, "NN", "f16", "normal", 1.0 / math.sqrt(4096), 2),
    "c4": Workload("square bf16 TN 8192^3", 8192, 8192, 8192, "TN", "bf16", "normal", 1.0 / math.sqrt(8192), 3),
    "c5": Workload("tall-skinny fp16 TN 16384x1024x8192", 16384, 1024, 8192, "TN", "f16", "uniform",
                   1.0 / math.sqrt(8192), 4),
    # 8-bit operands: the scaled contraction of the mma syntax page.
    "c4-e4m3": Workload("square E4M3 TN 8192^3, bf16 C, per-tensor scales", 8192, 8192, 8192, "TN", "e4m3",
                        "normal", 1.0, 5, out="bf16", scales="tensor"),
    "c4-mx": Workload("square E4M3 TN 8192^3, bf16 C, E8M0 scales per 32 K", 8192, 8192, 8192, "TN", "e4m3",
                      "normal", 1.0, 6, out="bf16", scales="block"),
    # A with a 2:4 pattern along K: the structured-sparsity form of the same page.
    "c4-sp": Workload("square bf16 TN 8192^3, A 2:4-sparse", 8192, 8192, 8192, "TN", "bf16", "normal",
                      1.0 / math.sqrt(4096), 7, sparse=True),
}


def prune_24(A: torch.Tensor, seed: int) -> torch.Tensor:
    """A copy of A (M x K, K % 4 == 0) with a 2:4 pattern along K: in every group of four
    consecutive elements of a row, two positions drawn uniformly from the six pairs (numpy
    generator seeded with `seed`) keep their values and the other two become zero."""
    import numpy as np

    M, K = A.shape
    if K % 4:
        raise ValueError("K must be a multiple of 4")
    pairs = np.array([[1, 1, 0, 0], [1, 0, 1, 0], [1, 0, 0, 1], [0, 1, 1, 0], [0, 1, 0, 1], [0, 0, 1, 1]], dtype=bool)
    rng = np.random.default_rng(seed)
    mask = pairs[rng.integers(0, 6, (M, K // 4))].reshape(M, K)
    out = A.clone()
    out[torch.from_numpy(~mask)] = 0
    return out


def tensor_scales(w: Workload):
    """Per-tensor scales of an 8-bit workload: K^-1/4 each, so C is of unit size."""
    s = float(w.K) ** -0.25
    return s, s


def block_scales(w: Workload):
    """(sa, sb): E8M0 exponents, M x ceil(K/32) and N x ceil(K/32) uint8 numpy arrays."""
    import numpy as np

    rng = np.random.default_rng(w.seed + 1000)
    nb = -(-w.K // 32)
    return (rng.integers(124, 131, (w.M, nb)).astype(np.uint8), rng.integers(124, 131, (w.N, nb)).astype(np.uint8))


def stored_b_shape(M: int, N: int, K: int, layout: str):
    return (K, N) if layout == "NN" else (N, K)


def _draw(gen: torch.Generator, shape, dist: str) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2 - 1
    if dist == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32)
    if dist == "int":
        return torch.randint(-2, 3, shape, generator=gen).to(torch.float32)
    if dist == "ones":
        return torch.ones(shape, dtype=torch.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def _padded(x: torch.Tensor, ld: int | None) -> torch.Tensor:
    rows, cols = x.shape
    if ld is None or ld == cols:
        return x.contiguous()
    if ld < cols:
        raise ValueError(f"leading dimension {ld} < row length {cols}")
    buf = torch.full((rows, ld), float("nan"), dtype=torch.float32).to(x.dtype)
    buf[:, :cols] = x
    return buf[:, :cols]


def make_inputs(M: int, N: int, K: int, layout: str, dtype: str, dist: str, seed: int,
                scale: float = 1.0, lda: int | None = None, ldb: int | None = None):
    """(A, B) as CPU tensors of the storage dtype; A is M x K, B its stored shape.

    With ``lda``/``ldb`` the tensors are views into NaN-padded row-major buffers.
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed))
    tdt = TORCH_DTYPES[dtype]
    a = _draw(gen, (M, K), dist)
    b = _draw(gen, stored_b_shape(M, N, K, layout), dist)
    if scale != 1.0:
        a = a * scale
        b = b * scale
    return _padded(a.to(tdt), lda), _padded(b.to(tdt), ldb)


def workload_inputs(w: Workload, lda: int | None = None, ldb: int | None = None):
    A, B = make_inputs(w.M, w.N, w.K, w.layout, w.dtype, w.dist, w.seed, w.scale, lda, ldb)
    if w.sparse:
        A = prune_24(A, w.seed + 2000)
    return A, B


def round_up(x: int, m: int) -> int:
    return -(-x // m) * m

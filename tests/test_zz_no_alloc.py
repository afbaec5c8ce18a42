"""gemm_run_noalloc: the entry point for callers that cannot allocate device memory.

Some callers may not call cudaMalloc at all -- plug-ins inside an engine that owns all
device memory, paths that cannot take the synchronisation an allocation may imply, a
process already at its memory limit.  For them the library keeps the kernel's only scratch
(its 16-byte watchdog record) in a static device array, so this entry point needs no handle
and allocates nothing.

The tests call it through the C ABI, always twice in a row, and compare every element with
the CPU oracle: bit for bit on integer-valued inputs in {-2..2} (ragged shapes in both
layouts and both 16-bit types, a problem large enough for the CTA pair, and one where
gemm_run splits K blocks between CTAs while this entry point takes whole tiles), and within
the parity tolerance on normal inputs.  Sentinel columns and rows around C must stay
untouched.  The file is collected last and passes both alone in a fresh process and after
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from dense_tiled_gemm_04_gb300 import native
from dense_tiled_gemm_04_gb300.workloads import make_inputs

import oracle

pytestmark = pytest.mark.gpu

TOL = {"f16": (1e-2, 1e-2), "bf16": (3e-2, 3e-2)}
SENTINEL = 0x7777  # a finite 16-bit code no product here produces
GUARD_ROWS, GUARD_COLS = 3, 8


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_tiled_gemm_04_gb300 import build

    build.build()
    oracle.build()
    torch.cuda.set_device(0)
    return native.load()


def _pad8(x: int) -> int:
    return -(-x // 8) * 8


def _device(x: torch.Tensor) -> torch.Tensor:
    """A CPU view (row pitch a multiple of 8 elements, NaN padding) copied to the GPU with its pitch."""
    rows, cols = x.shape
    base = x.as_strided((rows, x.stride(0)), (x.stride(0), 1))
    return base.cuda()[:, :cols]


def _codes(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _inputs(M, N, K, layout, dtype, dist, seed):
    return make_inputs(M, N, K, layout, dtype, dist, seed=seed, lda=_pad8(K) + 8,
                       ldb=_pad8(N if layout == "NN" else K) + 8)


def _run_noalloc(lib, A, B, M, N, K, layout, dtype, stream):
    """One gemm_run_noalloc call into a sentinel-filled buffer; returns (C codes, whole buffer codes)."""
    dA, dB = _device(A), _device(B)
    ldc = _pad8(N) + GUARD_COLS
    buf = torch.full((M + GUARD_ROWS, ldc), SENTINEL, dtype=torch.int16, device="cuda").view(A.dtype)
    C = buf[:M, :N]
    info = (ctypes.c_int32 * 4)(7, 7, 7, 7)
    st = lib.gemm_run_noalloc(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, dA.stride(0), dB.stride(0), ldc,
                              native.LAYOUTS[layout], native.DTYPES[dtype], stream.cuda_stream, info)
    assert st == native.OK, native.status_string(st)
    assert list(info) == [0, 0, 0, 0]  # the watchdog record was cleared and stayed clear
    return _codes(C), _codes(buf)


def _guard_intact(buf: np.ndarray, M: int, N: int):
    assert (buf[M:, :] == SENTINEL).all(), "rows below C were written"
    assert (buf[:, N:] == SENTINEL).all(), "columns right of C were written"


@pytest.mark.parametrize("first,second", [
    ((777, 1333, 515, "NN", "bf16"), (1000, 1000, 1000, "TN", "f16")),
    ((65, 97, 130, "TN", "bf16"), (300, 1, 77, "NN", "f16")),
    ((129, 257, 65, "NN", "f16"), (255, 511, 200, "TN", "bf16")),
])
def test_noalloc_is_bit_exact_on_integers_two_calls_in_a_row(lib, first, second):
    stream = torch.cuda.current_stream()
    for seed, (M, N, K, layout, dtype) in enumerate((first, second)):
        A, B = _inputs(M, N, K, layout, dtype, "int", 60 + seed)
        got, buf = _run_noalloc(lib, A, B, M, N, K, layout, dtype, stream)
        want = oracle.gemm(A, B, layout, dtype)
        assert np.array_equal(got, want), f"call {seed + 1}: {(got != want).sum()} codes differ from the oracle"
        _guard_intact(buf, M, N)


def test_noalloc_whole_tiles_equal_gemm_runs_split_k_and_the_oracle(lib):
    # A problem where the handle's gemm_run takes the CTA pair and shares the K blocks of
    # part-empty waves between pairs (stream-K); gemm_run_noalloc runs the same kernel on
    # whole tiles.  On integers both must equal the oracle bit for bit, hence each other.
    stream = torch.cuda.current_stream()
    M, N, K = 3072, 3072, 2048
    handle = native.Gemm(0)
    try:
        for seed, (layout, dtype) in enumerate((("TN", "bf16"), ("NN", "f16"))):
            plan = handle.plan(M, N, K, layout, dtype)
            assert plan["cluster"] == 2 and plan["sk_base"] > 0 and plan["dp_tiles"] < plan["tiles_m"] * plan["tiles_n"]
            A, B = _inputs(M, N, K, layout, dtype, "int", 70 + seed)
            got, buf = _run_noalloc(lib, A, B, M, N, K, layout, dtype, stream)
            dA, dB = _device(A), _device(B)
            ref = native.empty_output(M, N, A.dtype, "cuda")
            st = handle.run_raw(dA.data_ptr(), dB.data_ptr(), ref.data_ptr(), M, N, K, dA.stride(0), dB.stride(0),
                                ref.stride(0), native.LAYOUTS[layout], native.DTYPES[dtype], stream.cuda_stream)
            assert st == native.OK and handle.sync_status(stream) == native.OK
            want = oracle.gemm(A, B, layout, dtype)
            assert np.array_equal(got, want), f"{layout} {dtype}: {(got != want).sum()} codes differ from the oracle"
            assert np.array_equal(_codes(ref), got)
            _guard_intact(buf, M, N)
    finally:
        handle.close()


def test_noalloc_within_tolerance_on_normal_inputs_two_calls_in_a_row(lib):
    stream = torch.cuda.current_stream()
    for seed, (M, N, K, layout, dtype) in enumerate(((1000, 1000, 1000, "TN", "f16"), (777, 1333, 515, "NN", "bf16"))):
        A, B = _inputs(M, N, K, layout, dtype, "normal", 40 + seed)
        got, buf = _run_noalloc(lib, A, B, M, N, K, layout, dtype, stream)
        g, r = oracle.decode(got, dtype), oracle.decode(oracle.gemm(A, B, layout, dtype), dtype)
        atol, rtol = TOL[dtype]
        bad = ~(np.abs(g - r) <= atol + rtol * np.abs(r))
        assert not bad.any(), f"call {seed + 1}: {bad.sum()} elements outside tolerance"
        _guard_intact(buf, M, N)


def test_noalloc_rejects_bad_arguments_like_gemm_run(lib):
    # Argument checks happen before any device work.
    assert lib.gemm_run_noalloc(None, None, None, 8, 8, 8, 8, 8, 8, 0, 0, None, None) == native.ERR_INVALID_ARG
    assert lib.gemm_run_noalloc(16, 16, 16, -1, 8, 8, 8, 8, 8, 0, 0, None, None) == native.ERR_INVALID_ARG
    assert lib.gemm_run_noalloc(18, 16, 16, 8, 8, 8, 8, 8, 8, 0, 0, None, None) == native.ERR_UNSUPPORTED

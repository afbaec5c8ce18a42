"""gemm_run_noalloc: the entry point for callers that cannot allocate device memory.

Some callers may not call cudaMalloc at all -- plug-ins inside an engine that owns all
device memory, paths that cannot take the synchronisation an allocation may imply, a
process already at its memory limit.  For them the library keeps the
kernel's only scratch (its 16-byte watchdog record) in a static device array, so this
entry point needs no handle and allocates nothing.

The test calls it through the C ABI twice in a row, on two different problems, and
checks each result against gemm_run's (the handle-based entry point) within the same
tolerance the parity tests use.  It lives in its own file, collected last, and passes
both alone in a fresh process and after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from dense_tiled_gemm_04_gb300 import native
from dense_tiled_gemm_04_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu

TOL = {"f16": (1e-2, 1e-2), "bf16": (3e-2, 3e-2)}


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_tiled_gemm_04_gb300 import build

    build.build()
    return native.load()


def _values(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("first,second", [
    ((1000, 1000, 1000, "TN", "f16"), (777, 1333, 515, "NN", "bf16")),
])
def test_noalloc_matches_gemm_run_on_two_calls_in_a_row(lib, first, second):
    torch.cuda.set_device(0)
    handle = native.Gemm(0)
    stream = torch.cuda.current_stream()
    try:
        for seed, (M, N, K, layout, dtype) in enumerate((first, second)):
            A, B = make_inputs(M, N, K, layout, dtype, "normal", seed=40 + seed,
                               lda=-(-K // 8) * 8, ldb=-(-(N if layout == "NN" else K) // 8) * 8)
            rows_b = B.shape[0]
            dA = A.as_strided((M, A.stride(0)), (A.stride(0), 1)).cuda()[:, :K]
            dB = B.as_strided((rows_b, B.stride(0)), (B.stride(0), 1)).cuda()[:, :B.shape[1]]
            ref = native.empty_output(M, N, A.dtype, "cuda")
            out = native.empty_output(M, N, A.dtype, "cuda")
            out.fill_(float("nan"))
            ld = (dA.stride(0), dB.stride(0), out.stride(0))

            st = handle.run_raw(dA.data_ptr(), dB.data_ptr(), ref.data_ptr(), M, N, K, *ld,
                                native.LAYOUTS[layout], native.DTYPES[dtype], stream.cuda_stream)
            assert st == native.OK, native.status_string(st)
            assert handle.sync_status(stream) == native.OK

            info = (ctypes.c_int32 * 4)(7, 7, 7, 7)
            st = lib.gemm_run_noalloc(dA.data_ptr(), dB.data_ptr(), out.data_ptr(), M, N, K, *ld,
                                      native.LAYOUTS[layout], native.DTYPES[dtype], stream.cuda_stream, info)
            assert st == native.OK, native.status_string(st)
            assert list(info) == [0, 0, 0, 0]  # the watchdog record was cleared and stayed clear

            got, want = _values(out), _values(ref)
            atol, rtol = TOL[dtype]
            assert np.isfinite(got).all()
            bad = ~(np.abs(got - want) <= atol + rtol * np.abs(want))
            assert not bad.any(), f"call {seed + 1}: {bad.sum()} elements outside tolerance"
    finally:
        handle.close()


def test_noalloc_rejects_bad_arguments_like_gemm_run(lib):
    # Argument checks happen before any device work.
    assert lib.gemm_run_noalloc(None, None, None, 8, 8, 8, 8, 8, 8, 0, 0, None, None) == native.ERR_INVALID_ARG
    assert lib.gemm_run_noalloc(16, 16, 16, -1, 8, 8, 8, 8, 8, 0, 0, None, None) == native.ERR_INVALID_ARG
    assert lib.gemm_run_noalloc(18, 16, 16, 8, 8, 8, 8, 8, 8, 0, 0, None, None) == native.ERR_UNSUPPORTED

"""GPU parity of the general epilogue (gemm_run_ex): C = alpha * A·B + beta * C, with C stored
row-major or column-major.

Integer inputs with small integer alpha/beta keep every intermediate exact, so results must
match the oracle bit for bit; random inputs with fractional alpha/beta are compared within
the usual tolerance.  C lives in a sentinel-filled buffer with spare rows and columns that
must stay untouched.
"""
import numpy as np
import pytest
import torch

from dense_tiled_gemm_04_gb300 import native
from dense_tiled_gemm_04_gb300.workloads import WORKLOADS, make_inputs, round_up, workload_inputs

import oracle
from test_gpu_parity import SENTINEL, assert_close, assert_exact, to_device

pytestmark = pytest.mark.gpu

NAN = {"f16": 0x7E00, "bf16": 0x7FC0}


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_tiled_gemm_04_gb300 import build

    build.build()
    oracle.build()
    h = native.Gemm(0)
    yield h
    h.close()


def run_ex(g, A, B, layout, dtype, alpha, beta, col_major, c_init=None, pad=8, extra=2):
    """gemm_run_ex through the C ABI.  c_init: logical M x N codes to start C from (None: NaN
    in the window when beta == 0, else required).  Returns (logical result codes M x N,
    whole storage buffer codes, storage shape of the logical window)."""
    M, K = A.shape
    N = B.shape[1] if layout == "NN" else B.shape[0]
    rows, cols = (N, M) if col_major else (M, N)          # storage: rows x cols, row-major
    ldc = round_up(max(cols, 1), 8) + pad
    buf = torch.full((rows + extra, ldc), 0, dtype=torch.int16)
    buf.fill_(SENTINEL)
    window = buf[:rows, :cols]
    logical = window.t() if col_major else window           # logical M x N view of the storage
    if c_init is None:
        logical.fill_(NAN[dtype] - 65536 if NAN[dtype] > 32767 else NAN[dtype])
    else:
        logical.copy_(torch.from_numpy(c_init.view(np.int16)))
    dbuf = buf.cuda()
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    dA, dB = to_device(A), to_device(B)
    lda = dA.stride(0) if M > 1 else round_up(max(K, 1), 8)
    ldb = dB.stride(0) if B.shape[0] > 1 else round_up(max(B.shape[1], 1), 8)
    st = g.run_ex_raw(dA.data_ptr(), dB.data_ptr(), dbuf.data_ptr(), M, N, K, lda, ldb, ldc, native.LAYOUTS[layout],
                      native.DTYPES[dtype], alpha, beta, int(col_major), 0)
    assert st == native.OK, native.status_string(st)
    assert g.sync_status() == native.OK
    out = dbuf.cpu().numpy().view(np.uint16)
    win = out[:rows, :cols]
    res = np.ascontiguousarray(win.T if col_major else win)
    return res, out, (rows, cols)


def guard_ok(out, rows, cols):
    guard = out.copy()
    guard[:rows, :cols] = SENTINEL
    return np.all(guard == SENTINEL)


def int_codes(M, N, dtype, seed):
    c, _ = make_inputs(M, N, N, "NN", dtype, "int", seed=seed)
    return c.view(torch.int16).numpy().view(np.uint16)


SHAPES = [(65, 97, 130), (300, 257, 200), (1000, 1000, 520), (1003, 131, 77)]


@pytest.mark.parametrize("col_major", [0, 1])
@pytest.mark.parametrize("config", [native.CONFIG_AUTO, native.CONFIG_128x256, native.CONFIG_128x64,
                                    native.CONFIG_256x256])
@pytest.mark.parametrize("layout,dtype", [("NN", "f16"), ("TN", "bf16"), ("TN", "f16"), ("NN", "bf16")])
def test_alpha_beta_and_layout(g, col_major, config, layout, dtype):
    g.set_option(native.OPT_CONFIG, config)
    try:
        for i, (M, N, K) in enumerate(SHAPES):
            bcols = N if layout == "NN" else K
            # integer data, integer scalars: exact
            A, B = make_inputs(M, N, K, layout, dtype, "int", seed=70 + i, lda=round_up(K, 8),
                               ldb=round_up(bcols, 8))
            C0 = int_codes(M, N, dtype, 80 + i)
            got, out, (r, c) = run_ex(g, A, B, layout, dtype, 2.0, -1.0, col_major, C0)
            assert guard_ok(out, r, c), "write outside the C window"
            assert_exact(got, oracle.gemm_axpby(A, B, layout, dtype, 2.0, -1.0, C0), f"{(M, N, K)} int a=2 b=-1")
            # random data, fractional scalars: tolerance
            A, B = make_inputs(M, N, K, layout, dtype, "normal", seed=90 + i, lda=round_up(K, 8),
                               ldb=round_up(bcols, 8))
            C0r, _ = make_inputs(M, N, N, "NN", dtype, "normal", seed=95 + i)
            C0r = C0r.view(torch.int16).numpy().view(np.uint16)
            got, out, (r, c) = run_ex(g, A, B, layout, dtype, 0.5, 1.5, col_major, C0r)
            assert guard_ok(out, r, c)
            assert_close(got, oracle.gemm_axpby(A, B, layout, dtype, 0.5, 1.5, C0r), dtype, f"{(M, N, K)} a=.5 b=1.5")
    finally:
        g.set_option(native.OPT_CONFIG, native.CONFIG_AUTO)


@pytest.mark.parametrize("col_major", [0, 1])
def test_beta_zero_never_reads_c(g, col_major):
    # C starts as NaN: with beta == 0 it must not be read, so no NaN may reach the result.
    M, N, K = 513, 300, 260
    A, B = make_inputs(M, N, K, "TN", "f16", "int", seed=5)
    got, out, (r, c) = run_ex(g, A, B, "TN", "f16", 1.0, 0.0, col_major, None)
    assert_exact(got, oracle.gemm(A, B, "TN", "f16"), "beta = 0 over NaN")
    assert guard_ok(out, r, c)


@pytest.mark.parametrize("col_major", [0, 1])
def test_column_major_equals_transposed_row_major(g, col_major):
    M, N, K = 777, 1029, 300
    A, B = make_inputs(M, N, K, "NN", "bf16", "int", seed=6, lda=round_up(K, 8), ldb=round_up(N, 8))
    got, _, _ = run_ex(g, A, B, "NN", "bf16", 1.0, 0.0, col_major, None)
    assert_exact(got, oracle.gemm(A, B, "NN", "bf16"), f"col_major={col_major}")


@pytest.mark.parametrize("col_major", [0, 1])
def test_k_zero_scales_c(g, col_major):
    M, N = 45, 70
    A = torch.empty((M, 0), dtype=torch.float16)
    B = torch.empty((0, N), dtype=torch.float16)
    C0 = int_codes(M, N, "f16", 7)
    got, out, (r, c) = run_ex(g, A, B, "NN", "f16", 3.0, -2.0, col_major, C0)
    assert guard_ok(out, r, c)
    assert_exact(got, oracle.encode(-2.0 * oracle.decode(C0, "f16"), "f16"), "K=0: C = beta C")


@pytest.mark.parametrize("config", [native.CONFIG_128x128, native.CONFIG_256x256])
@pytest.mark.parametrize("col_major", [0, 1])
def test_stream_k_with_epilogue(g, config, col_major):
    M, N, K = 1000, 1000, 2048
    A, B = make_inputs(M, N, K, "TN", "bf16", "int", seed=8)
    C0 = int_codes(M, N, "bf16", 9)
    g.set_option(native.OPT_CONFIG, config)
    g.set_option(native.OPT_MAX_CTAS, 12)
    try:
        pl = g.plan(M, N, K, "TN", "bf16")
        assert pl["dp_tiles"] < pl["tiles_m"] * pl["tiles_n"], "stream-K not engaged"
        got, out, (r, c) = run_ex(g, A, B, "TN", "bf16", -1.0, 2.0, col_major, C0)
    finally:
        g.set_option(native.OPT_CONFIG, native.CONFIG_AUTO)
        g.set_option(native.OPT_MAX_CTAS, 0)
    assert guard_ok(out, r, c)
    assert_exact(got, oracle.gemm_axpby(A, B, "TN", "bf16", -1.0, 2.0, C0), "stream-K + epilogue")


def test_full_size_column_major_accumulate(g):
    # The headline shape, C += A·B into a column-major C: every element against the oracle.
    w = WORKLOADS["c4"].with_dist("int")
    A, B = workload_inputs(w)
    C0 = int_codes(w.M, w.N, "bf16", 10)
    got, _, _ = run_ex(g, A, B, w.layout, "bf16", 1.0, 1.0, 1, C0, pad=0, extra=0)
    ref = oracle.gemm_axpby(A, B, w.layout, "bf16", 1.0, 1.0, C0)
    assert_exact(got, ref, "c4 C += A·B, column-major")


def test_invalid_epilogue_arguments(g):
    buf = torch.zeros((64, 64), dtype=torch.float16, device="cuda")
    p = buf.data_ptr()
    assert g.run_ex_raw(p, p, p, 64, 64, 64, 64, 64, 64, 0, 0, 1.0, 0.0, 2, 0) == native.ERR_INVALID_ARG
    assert g.run_ex_raw(p, p, p, 64, 64, 64, 64, 64, 64, 0, 0, float("nan"), 0.0, 0, 0) == native.ERR_INVALID_ARG
    # column-major C needs ldc >= M
    assert g.run_ex_raw(p, p, p, 72, 64, 64, 64, 64, 64, 0, 0, 1.0, 0.0, 1, 0) == native.ERR_INVALID_ARG
    assert g.sync_status() == native.OK

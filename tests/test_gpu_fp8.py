"""GPU parity of 8-bit float operands (E4M3, E5M2) with per-tensor scales, through gemm_run_ex.

The operation is the scaled form of the contraction in "张量缩并：mma 语法": C = alpha *
scale_a * scale_b * (A·B) + beta * C with A, B 8-bit floats, the products accumulated in
fp32 and C rounded once to fp16 or bf16.

Bar: integer-valued operands in {-2..2} (exact in both 8-bit formats) with power-of-two
alpha, scales and beta keep every intermediate exact in fp32, so the result must match the
oracle bit for bit; normal operands with fractional scales are compared within
|gpu - ref| <= atol + rtol * |ref|, atol = rtol = 1e-2 (fp16 C) or 3e-2 (bf16 C): every
product of two 8-bit floats is exact in fp32, the fp32 sum of K <= 8192 terms is off by
at most ~K * 2^-24 relative to the sum of magnitudes, and the one rounding to the output
type adds half an ulp (2^-11 for fp16, 2^-8 for bf16).
"""
import numpy as np
import pytest
import torch

from dense_tiled_gemm_04_gb300 import native
from dense_tiled_gemm_04_gb300.workloads import make_inputs, round_up

import oracle
from test_gpu_parity import SENTINEL, assert_close, assert_exact

pytestmark = pytest.mark.gpu

OUT_TORCH = {"f16": torch.float16, "bf16": torch.bfloat16}
NAN16 = {"f16": 0x7E00, "bf16": 0x7FC0}


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


def to_device8(x: torch.Tensor) -> torch.Tensor:
    """Copy a (possibly row-padded) 8-bit CPU view to the GPU keeping its row pitch; a row
    pitch that is not a multiple of 16 elements is widened to one (NaN padding)."""
    rows, cols = x.shape
    if rows > 1 and x.stride(0) % 16 != 0:
        buf = torch.full((rows, round_up(cols, 16)), float("nan")).to(x.dtype)
        buf.view(torch.uint8)[:, :cols] = x.view(torch.uint8)
        x = buf[:, :cols]
    ld = x.stride(0) if rows > 1 else round_up(max(cols, 1), 16)
    if rows > 1:
        base = x.as_strided((rows, ld), (ld, 1))
    else:
        base = torch.full((rows, ld), float("nan")).to(x.dtype)
        base.view(torch.uint8)[:, :cols] = x.view(torch.uint8)
    return base.cuda()[:, :cols]


def run8(g, A, B, layout, out, alpha=1.0, beta=0.0, scale_a=1.0, scale_b=1.0, col_major=False, c_init=None,
         pad=8, extra=2):
    """gemm_run_ex with 8-bit A, B.  C starts from c_init (logical M x N codes) or, with
    beta == 0, NaN; it sits in a sentinel-filled buffer with spare rows and columns.
    Returns (logical result codes M x N, True if the guard region is untouched)."""
    M, K = A.shape
    N = B.shape[1] if layout == "NN" else B.shape[0]
    rows, cols = (N, M) if col_major else (M, N)
    ldc = round_up(max(cols, 1), 8) + pad
    buf = torch.full((rows + extra, ldc), 0, dtype=torch.int16)
    buf.fill_(SENTINEL)
    window = buf[:rows, :cols]
    logical = window.t() if col_major else window
    if c_init is None:
        logical.fill_(NAN16[out] - 65536 if NAN16[out] > 32767 else NAN16[out])
    else:
        logical.copy_(torch.from_numpy(c_init.view(np.int16)))
    dbuf = buf.cuda()
    dA, dB = to_device8(A), to_device8(B)
    lda = dA.stride(0) if M > 1 else round_up(max(K, 1), 16)
    ldb = dB.stride(0) if B.shape[0] > 1 else round_up(max(B.shape[1], 1), 16)
    st = g.run_ex_raw(dA.data_ptr(), dB.data_ptr(), dbuf.data_ptr(), M, N, K, lda, ldb, ldc, native.LAYOUTS[layout],
                      native.TORCH_TO_DTYPE_EX[A.dtype], alpha, beta, int(col_major), 0, native.DTYPES[out],
                      scale_a, scale_b)
    assert st == native.OK, native.status_string(st)
    assert g.sync_status() == native.OK
    res = dbuf.cpu().numpy().view(np.uint16)
    win = res[:rows, :cols]
    guard = res.copy()
    guard[:rows, :cols] = SENTINEL
    return np.ascontiguousarray(win.T if col_major else win), bool(np.all(guard == SENTINEL))


def factor(alpha, scale_a, scale_b) -> float:
    """The fp32 product the library documents: (alpha * scale_a) * scale_b in fp32."""
    return float(np.float32(np.float32(alpha) * np.float32(scale_a)) * np.float32(scale_b))


def int_c(M, N, out, seed):
    c, _ = make_inputs(M, N, N, "NN", out, "int", seed=seed)
    return c.view(torch.int16).numpy().view(np.uint16)


CONFIGS = [native.CONFIG_AUTO, native.CONFIG_128x256, native.CONFIG_128x128, native.CONFIG_256x256,
           native.CONFIG_128x64]  # 128x64 runs 128x128 for 8-bit operands
IN_TYPES = ["e4m3", "e5m2"]


@pytest.fixture
def config(g, request):
    g.set_option(native.OPT_CONFIG, request.param)
    yield request.param
    g.set_option(native.OPT_CONFIG, native.CONFIG_AUTO)


@pytest.mark.parametrize("config", CONFIGS, indirect=True)
@pytest.mark.parametrize("layout", ["NN", "TN"])
@pytest.mark.parametrize("in_dtype", IN_TYPES)
@pytest.mark.parametrize("out", ["f16", "bf16"])
def test_int_operands_bit_exact(g, config, layout, in_dtype, out):
    # Ragged in M, N and K (K = 4 stages of 128 + 8), power-of-two factors.
    M, N, K = 300, 257, 520
    A, B = make_inputs(M, N, K, layout, in_dtype, "int", seed=11)
    got, guard = run8(g, A, B, layout, out, alpha=0.25, scale_a=0.5, scale_b=2.0)
    ref = oracle.gemm_typed(A, B, layout, in_dtype, out, alpha=factor(0.25, 0.5, 2.0))
    assert guard
    assert_exact(got, ref, f"{in_dtype}->{out} {layout} config {config}")


@pytest.mark.parametrize("config", CONFIGS, indirect=True)
@pytest.mark.parametrize("layout", ["NN", "TN"])
@pytest.mark.parametrize("in_dtype", IN_TYPES)
def test_normal_operands_within_tolerance(g, config, layout, in_dtype):
    M, N, K = 515, 389, 1000
    A, B = make_inputs(M, N, K, layout, in_dtype, "normal", seed=12)
    sa, sb = 1.0 / 5.3, 1.0 / 6.1  # ~ K^-1/4 each: the results are of unit size
    for out in ("f16", "bf16"):
        got, guard = run8(g, A, B, layout, out, scale_a=sa, scale_b=sb)
        ref = oracle.gemm_typed(A, B, layout, in_dtype, out, alpha=factor(1.0, sa, sb))
        assert guard
        assert_close(got, ref, out, f"{in_dtype}->{out} {layout} config {config}")


@pytest.mark.parametrize("col_major", [False, True])
@pytest.mark.parametrize("layout", ["NN", "TN"])
@pytest.mark.parametrize("in_dtype", IN_TYPES)
def test_accumulate_and_column_major_bit_exact(g, col_major, layout, in_dtype):
    M, N, K = 333, 200, 264
    A, B = make_inputs(M, N, K, layout, in_dtype, "int", seed=13)
    for out in ("f16", "bf16"):
        c0 = int_c(M, N, out, seed=14)
        got, guard = run8(g, A, B, layout, out, alpha=2.0, beta=-0.5, scale_a=1.0, scale_b=0.5, col_major=col_major,
                          c_init=c0)
        ref = oracle.gemm_typed(A, B, layout, in_dtype, out, alpha=factor(2.0, 1.0, 0.5), beta=-0.5, Cin=c0)
        assert guard
        assert_exact(got, ref, f"{in_dtype}->{out} {layout} col_major={col_major}")


@pytest.mark.parametrize("shape", [(1, 1, 1), (7, 9, 16), (128, 256, 128), (129, 257, 129), (64, 48, 40),
                                   (256, 256, 4096), (3, 600, 31)])
@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_edge_shapes(g, shape, layout):
    M, N, K = shape
    A, B = make_inputs(M, N, K, layout, "e4m3", "int", seed=15)
    got, guard = run8(g, A, B, layout, "bf16")
    ref = oracle.gemm_typed(A, B, layout, "e4m3", "bf16")
    assert guard
    assert_exact(got, ref, f"{shape} {layout}")


@pytest.mark.parametrize("out", ["f16", "bf16"])
def test_k_zero_scales_c(g, out):
    M, N = 70, 45
    A = torch.zeros((M, 0)).to(torch.float8_e4m3fn)
    B = torch.zeros((0, N)).to(torch.float8_e4m3fn)
    c0 = int_c(M, N, out, seed=16)
    dbuf = torch.from_numpy(c0.view(np.int16).copy())
    dC = torch.zeros((M, round_up(N, 8)), dtype=torch.int16, device="cuda")
    dC[:, :N] = dbuf.cuda()
    st = g.run_ex_raw(16, 16, dC.data_ptr(), M, N, 0, 16, 64, dC.stride(0), native.LAYOUT_NN, native.DTYPE_E4M3,
                      1.0, 3.0, 0, 0, native.DTYPES[out], 0.5, 0.5)
    assert st == native.OK
    assert g.sync_status() == native.OK
    got = dC[:, :N].cpu().numpy().view(np.uint16)
    ref = oracle.encode(3.0 * oracle.decode(c0, out), out)
    assert_exact(got, ref, "K == 0")


@pytest.mark.parametrize("in_dtype", IN_TYPES)
@pytest.mark.parametrize("stream_k,k_snake", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_multi_tile_stream_k_bit_exact(g, in_dtype, stream_k, k_snake):
    # 16384 x 1024 tiles leave the last wave part-empty: stream-K shares its K blocks out.
    M, N, K = 16384, 1024, 2048
    A, B = make_inputs(M, N, K, "TN", in_dtype, "int", seed=17)
    snake0 = g.get_option(native.OPT_K_SNAKE)
    g.set_option(native.OPT_STREAM_K, stream_k)
    g.set_option(native.OPT_K_SNAKE, k_snake)
    try:
        plan = g.plan(M, N, K, "TN", in_dtype)
        assert plan["bk"] == 128 and plan["k_blocks"] == K // 128
        if stream_k:
            assert plan["dp_tiles"] < plan["tiles_m"] * plan["tiles_n"]
        dA, dB = to_device8(A), to_device8(B)
        C = g.run_ex(dA, dB, layout="TN", out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        assert g.sync_status() == native.OK
    finally:
        g.set_option(native.OPT_STREAM_K, 1)
        g.set_option(native.OPT_K_SNAKE, snake0)
    got = C.cpu().view(torch.int16).numpy().view(np.uint16)
    ref = oracle.gemm_typed(A, B, "TN", in_dtype, "bf16")
    assert_exact(got, ref, f"{in_dtype} stream_k={stream_k} k_snake={k_snake}")


@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_full_size_e4m3_8192_full_matrix(g, layout):
    # The square 8192^3 problem with E4M3 operands (unit-normal draws, 1/sqrt(K) as the two
    # per-tensor scales), bf16 C, default plan.
    M = N = K = 8192
    A, B = make_inputs(M, N, K, layout, "e4m3", "normal", seed=19)
    s = K ** -0.25
    C = g.run_ex(to_device8(A), to_device8(B), layout=layout, out_dtype=torch.bfloat16, scale_a=s, scale_b=s)
    torch.cuda.synchronize()
    assert g.sync_status() == native.OK
    got = C.cpu().view(torch.int16).numpy().view(np.uint16)
    ref = oracle.gemm_typed(A, B, layout, "e4m3", "bf16", alpha=factor(1.0, s, s))
    assert_close(got, ref, "bf16", f"e4m3 8192^3 {layout}")


def test_run_ex_wrapper_matches_raw_call(g):
    M, N, K = 200, 136, 96
    A, B = make_inputs(M, N, K, "TN", "e5m2", "int", seed=21)
    C = g.run_ex(to_device8(A), to_device8(B), layout="TN", out_dtype=torch.float16, alpha=0.5)
    torch.cuda.synchronize()
    got = C.cpu().view(torch.int16).numpy().view(np.uint16)
    assert_exact(got, oracle.gemm_typed(A, B, "TN", "e5m2", "f16", alpha=0.5), "run_ex")


def test_invalid_arguments(g):
    A = torch.zeros((32, 32)).to(torch.float8_e4m3fn).cuda()
    B = torch.zeros((32, 32)).to(torch.float8_e4m3fn).cuda()
    C = torch.zeros((32, 32), dtype=torch.bfloat16, device="cuda")
    a, b, c = A.data_ptr(), B.data_ptr(), C.data_ptr()

    def ex(**kw):
        args = dict(M=32, N=32, K=32, lda=32, ldb=32, ldc=32, layout=0, dtype=native.DTYPE_E4M3, alpha=1.0, beta=0.0,
                    c_col_major=0, stream=0, out_dtype=native.DTYPE_BF16, scale_a=1.0, scale_b=1.0)
        args.update(kw)
        return g.run_ex_raw(a, b, c, args["M"], args["N"], args["K"], args["lda"], args["ldb"], args["ldc"],
                            args["layout"], args["dtype"], args["alpha"], args["beta"], args["c_col_major"],
                            args["stream"], args["out_dtype"], args["scale_a"], args["scale_b"])

    assert ex() == native.OK
    assert g.sync_status() == native.OK
    assert ex(lda=40, K=24) == native.ERR_UNSUPPORTED          # 8-bit pitch not a multiple of 16
    assert ex(ldb=40, N=24, ldc=32) == native.ERR_UNSUPPORTED
    assert ex(out_dtype=native.DTYPE_E4M3) == native.ERR_INVALID_ARG  # 8-bit output
    assert ex(out_dtype=7) == native.ERR_INVALID_ARG
    assert ex(dtype=native.DTYPE_F16, out_dtype=native.DTYPE_BF16) == native.ERR_INVALID_ARG  # 16-bit: out == in
    assert ex(scale_a=float("inf")) == native.ERR_INVALID_ARG
    assert ex(scale_b=float("nan")) == native.ERR_INVALID_ARG
    assert ex(alpha=3e38, scale_a=10.0) == native.ERR_INVALID_ARG  # the product overflows fp32
    # gemm_run takes 16-bit operands only.
    assert g.run_raw(a, b, c, 32, 32, 32, 32, 32, 32, 0, native.DTYPE_E4M3, 0) == native.ERR_INVALID_ARG

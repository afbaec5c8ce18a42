"""GPU parity of 8-bit operands with per-tile E8M0 scales (gemm_run_mx) against the oracle.

The scaled contraction of "张量缩并：mma 语法" with tiles of one row of A (one column of B)
by 32 K elements: acc = sum_j 2^(ea - 127) * 2^(eb - 127) * (A·B over K block j), then
C = alpha * scale_a * scale_b * acc + beta * C, rounded once to fp16 / bf16.

Bar: integer operands in {-2..2} with scale exponents within 2 of 127 keep every partial
sum a multiple of 2^-4 below 2^17 -- exact in fp32 in any order -- so the result must match
the oracle bit for bit; normal operands with exponents within 3 of 127 are compared within
atol = rtol = 1e-2 (fp16 C) / 3e-2 (bf16 C), as for the unscaled 8-bit path.
"""
import numpy as np
import pytest
import torch

from dense_tiled_gemm_04_gb300 import native
from dense_tiled_gemm_04_gb300.workloads import make_inputs, round_up

import oracle
from test_gpu_fp8 import factor, int_c, run8, to_device8
from test_gpu_parity import SENTINEL, assert_close, assert_exact

pytestmark = pytest.mark.gpu

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


# AUTO picks the CTA pair for large problems; 128x256 / 256x256 force the one-CTA tile / the pair.
CONFIGS = [native.CONFIG_AUTO, native.CONFIG_128x256, native.CONFIG_256x256]


@pytest.fixture
def config(g, request):
    g.set_option(native.OPT_CONFIG, request.param)
    yield request.param
    g.set_option(native.OPT_CONFIG, native.CONFIG_AUTO)


def scales(rows, K, spread, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(127 - spread, 128 + spread, (rows, -(-K // 32))).astype(np.uint8)


def packed(g, s: np.ndarray, K: int) -> torch.Tensor:
    return g.pack_scales(torch.from_numpy(s).cuda(), K)


def run_mx(g, A, B, sa, sb, layout, out, alpha=1.0, beta=0.0, scale_a=1.0, scale_b=1.0, col_major=False,
           c_init=None, pad=8, extra=2):
    """gemm_run_mx with C in a sentinel-filled buffer.  Returns (logical M x N codes, guard ok)."""
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
    psa, psb = packed(g, sa, K), packed(g, sb, K)
    st = g.run_mx_raw(dA.data_ptr(), dB.data_ptr(), dbuf.data_ptr(), psa.data_ptr(), psb.data_ptr(), M, N, K, lda,
                      ldb, ldc, native.LAYOUTS[layout], native.TORCH_TO_DTYPE_EX[A.dtype], native.DTYPES[out], alpha,
                      beta, int(col_major), scale_a, scale_b, 0)
    assert st == native.OK, native.status_string(st)
    assert g.sync_status() == native.OK
    res = dbuf.cpu().numpy().view(np.uint16)
    win = res[:rows, :cols]
    guard = res.copy()
    guard[:rows, :cols] = SENTINEL
    return np.ascontiguousarray(win.T if col_major else win), bool(np.all(guard == SENTINEL))


def expected_chunks(s: np.ndarray) -> np.ndarray:
    """The chunked layout written out from its definition: chunk (rb, g) at (rb * G + g) * 512,
    row r and K block c of the chunk at (r % 32) * 16 + (r // 32) * 4 + c, padding 127."""
    rows, kb = s.shape
    RB, G = -(-rows // 128), -(-kb // 4)
    out = np.full(RB * G * 512, 127, np.uint8)
    for r in range(rows):
        for j in range(kb):
            rb, rr, gg, c = r // 128, r % 128, j // 4, j % 4
            out[(rb * G + gg) * 512 + (rr % 32) * 16 + (rr // 32) * 4 + c] = s[r, j]
    return out


@pytest.mark.parametrize("rows,kb", [(1, 1), (128, 4), (300, 17), (129, 5), (64, 256)])
def test_pack_scales_layout(g, rows, kb):
    s = scales(rows, 32 * kb, 100, seed=rows + kb)
    got = packed(g, s, 32 * kb).cpu().numpy()
    assert got.size == native.mx_scale_bytes(rows, 32 * kb)
    assert np.array_equal(got, expected_chunks(s))


def test_scale_bytes():
    assert native.mx_scale_bytes(0, 64) == 0 and native.mx_scale_bytes(5, 0) == 0
    assert native.mx_scale_bytes(128, 128) == 512
    assert native.mx_scale_bytes(129, 129) == 2 * 2 * 512
    assert native.mx_scale_bytes(300, 8192) == 3 * 64 * 512


@pytest.mark.parametrize("config", CONFIGS[1:], indirect=True)
@pytest.mark.parametrize("layout", ["NN", "TN"])
@pytest.mark.parametrize("in_dtype", ["e4m3", "e5m2"])
@pytest.mark.parametrize("out", ["f16", "bf16"])
def test_int_operands_bit_exact(g, config, layout, in_dtype, out):
    M, N, K = 300, 600, 520  # ragged M, N (the last tile has one B scale chunk) and K (17 blocks)
    A, B = make_inputs(M, N, K, layout, in_dtype, "int", seed=61)
    sa, sb = scales(M, K, 2, seed=62), scales(N, K, 2, seed=63)
    got, guard = run_mx(g, A, B, sa, sb, layout, out, alpha=0.5, scale_a=2.0, scale_b=0.25)
    ref = oracle.gemm_blockscaled(A, B, sa, sb, layout, in_dtype, out, alpha=factor(0.5, 2.0, 0.25))
    assert guard
    assert_exact(got, ref, f"{in_dtype}->{out} {layout}")


@pytest.mark.parametrize("config", CONFIGS[1:], indirect=True)
@pytest.mark.parametrize("layout", ["NN", "TN"])
@pytest.mark.parametrize("in_dtype", ["e4m3", "e5m2"])
def test_normal_operands_within_tolerance(g, config, layout, in_dtype):
    M, N, K = 515, 389, 1000
    A, B = make_inputs(M, N, K, layout, in_dtype, "normal", seed=64)
    sa, sb = scales(M, K, 3, seed=65), scales(N, K, 3, seed=66)
    for out in ("f16", "bf16"):
        got, guard = run_mx(g, A, B, sa, sb, layout, out, scale_a=1 / 32, scale_b=1.0)
        ref = oracle.gemm_blockscaled(A, B, sa, sb, layout, in_dtype, out, alpha=factor(1.0, 1 / 32, 1.0))
        assert guard
        assert_close(got, ref, out, f"{in_dtype}->{out} {layout}")


def test_unit_scales_equal_the_unscaled_kernel(g):
    M, N, K = 256, 512, 384
    A, B = make_inputs(M, N, K, "TN", "e4m3", "normal", seed=67)
    one_a, one_b = np.full((M, K // 32), 127, np.uint8), np.full((N, K // 32), 127, np.uint8)
    got, _ = run_mx(g, A, B, one_a, one_b, "TN", "bf16")
    plain, _ = run8(g, A, B, "TN", "bf16")
    # Same products, same fp32 sums in one tile: any difference would be the scales.
    assert_close(got, plain, "bf16", "unit scales")
    assert_close(got, oracle.gemm_typed(A, B, "TN", "e4m3", "bf16"), "bf16", "unit scales vs oracle")


@pytest.mark.parametrize("config", CONFIGS[1:], indirect=True)
@pytest.mark.parametrize("col_major", [False, True])
@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_accumulate_and_column_major_bit_exact(g, config, col_major, layout):
    M, N, K = 333, 200, 264
    A, B = make_inputs(M, N, K, layout, "e4m3", "int", seed=68)
    sa, sb = scales(M, K, 2, seed=69), scales(N, K, 2, seed=70)
    for out in ("f16", "bf16"):
        c0 = int_c(M, N, out, seed=71)
        got, guard = run_mx(g, A, B, sa, sb, layout, out, alpha=2.0, beta=-0.5, col_major=col_major, c_init=c0)
        ref = oracle.gemm_blockscaled(A, B, sa, sb, layout, "e4m3", out, alpha=2.0, beta=-0.5, Cin=c0)
        assert guard
        assert_exact(got, ref, f"{out} {layout} col_major={col_major}")


@pytest.mark.parametrize("shape", [(1, 1, 1), (7, 9, 16), (128, 256, 128), (129, 257, 129), (64, 48, 40),
                                   (256, 256, 4096), (3, 600, 31)])
@pytest.mark.parametrize("config", CONFIGS[1:], indirect=True)
@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_edge_shapes(g, config, shape, layout):
    M, N, K = shape
    A, B = make_inputs(M, N, K, layout, "e5m2", "int", seed=72)
    sa, sb = scales(M, K, 2, seed=73), scales(N, K, 2, seed=74)
    got, guard = run_mx(g, A, B, sa, sb, layout, "f16")
    assert guard
    assert_exact(got, oracle.gemm_blockscaled(A, B, sa, sb, layout, "e5m2", "f16"), f"{shape} {layout}")


@pytest.mark.parametrize("config", CONFIGS[1:], indirect=True)
def test_one_block_scale_reaches_only_its_rows(g, config):
    # A NaN exponent in one K block of one row of A poisons exactly that row of C, in either
    # CTA's half of a pair tile; one of a column of B, exactly that column (in both halves).
    M, N, K = 256, 256, 256
    A, B = make_inputs(M, N, K, "TN", "e4m3", "int", seed=75)
    sa, sb = np.full((M, 8), 127, np.uint8), np.full((N, 8), 127, np.uint8)
    sa[77, 5] = 255
    sa[180, 1] = 255
    got, _ = run_mx(g, A, B, sa, sb, "TN", "bf16")
    vals = oracle.decode(got, "bf16")
    assert np.all(np.isnan(vals[[77, 180]]))
    assert not np.isnan(np.delete(vals, [77, 180], axis=0)).any()
    sa[77, 5] = sa[180, 1] = 127
    sb[200, 2] = 255
    sb[40, 7] = 255
    got, _ = run_mx(g, A, B, sa, sb, "TN", "bf16")
    vals = oracle.decode(got, "bf16")
    assert np.all(np.isnan(vals[:, [40, 200]]))
    assert not np.isnan(np.delete(vals, [40, 200], axis=1)).any()


@pytest.mark.parametrize("config", CONFIGS[1:], indirect=True)
@pytest.mark.parametrize("stream_k", [0, 1])
def test_multi_tile_stream_k_bit_exact(g, config, stream_k):
    M, N, K = 16384, 1024, 2048
    A, B = make_inputs(M, N, K, "TN", "e4m3", "int", seed=76)
    sa, sb = scales(M, K, 2, seed=77), scales(N, K, 2, seed=78)
    g.set_option(native.OPT_STREAM_K, stream_k)
    try:
        C = g.run_mx(to_device8(A), to_device8(B), packed(g, sa, K), packed(g, sb, K), layout="TN",
                     out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        assert g.sync_status() == native.OK
    finally:
        g.set_option(native.OPT_STREAM_K, 1)
    got = C.cpu().view(torch.int16).numpy().view(np.uint16)
    ref = oracle.gemm_blockscaled(A, B, sa, sb, "TN", "e4m3", "bf16")
    assert_exact(got, ref, f"stream_k={stream_k}")


@pytest.mark.parametrize("config", CONFIGS[1:], indirect=True)
@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_scale_ring_across_split_items_bit_exact(g, config, layout):
    # Scales travel in slots of four stages, counted from each work item's first K block: K of
    # 21 stages (a last slot of one stage) and few CTAs, so stream-K items start and end inside
    # slots and several items pass through the two-slot ring per CTA.
    M, N, K = 1000, 1000, 2600
    A, B = make_inputs(M, N, K, layout, "e4m3", "int", seed=87)
    sa, sb = scales(M, K, 2, seed=88), scales(N, K, 2, seed=89)
    # The option that reverses every second item's K order leaves block-scaled kernels alone.
    snake0 = g.get_option(native.OPT_K_SNAKE)
    g.set_option(native.OPT_MAX_CTAS, 10)
    g.set_option(native.OPT_K_SNAKE, 1)
    try:
        pl = g.plan(M, N, K, layout, "e4m3", "block_scaled")
        assert pl["k_blocks"] == 21 and pl["dp_tiles"] < pl["tiles_m"] * pl["tiles_n"], pl
        got, guard = run_mx(g, A, B, sa, sb, layout, "bf16")
    finally:
        g.set_option(native.OPT_MAX_CTAS, 0)
        g.set_option(native.OPT_K_SNAKE, snake0)
    assert guard
    assert_exact(got, oracle.gemm_blockscaled(A, B, sa, sb, layout, "e4m3", "bf16"), f"{layout}")


@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_full_size_8192_full_matrix(g, layout):
    M = N = K = 8192
    A, B = make_inputs(M, N, K, layout, "e4m3", "normal", seed=80)
    sa, sb = scales(M, K, 3, seed=81), scales(N, K, 3, seed=82)
    C = g.run_mx(to_device8(A), to_device8(B), packed(g, sa, K), packed(g, sb, K), layout=layout,
                 out_dtype=torch.bfloat16, scale_a=1 / 64, scale_b=1 / 64)
    torch.cuda.synchronize()
    assert g.sync_status() == native.OK
    got = C.cpu().view(torch.int16).numpy().view(np.uint16)
    ref = oracle.gemm_blockscaled(A, B, sa, sb, layout, "e4m3", "bf16", alpha=factor(1.0, 1 / 64, 1 / 64))
    assert_close(got, ref, "bf16", f"8192^3 {layout}")


@pytest.mark.parametrize("config", CONFIGS[1:], indirect=True)
def test_watchdog_reports_a_timeout(g, config):
    M, N, K = 512, 512, 1024
    A, B = make_inputs(M, N, K, "TN", "e4m3", "int", seed=84)
    sa, sb = scales(M, K, 2, seed=85), scales(N, K, 2, seed=86)
    dA, dB, psa, psb = to_device8(A), to_device8(B), packed(g, sa, K), packed(g, sb, K)
    g.set_option(native.OPT_TIMEOUT_NS, 20_000_000)
    g.set_option(native.OPT_FAULT_INJECT, 1)
    try:
        g.run_mx(dA, dB, psa, psb, layout="TN")
        assert g.sync_status() == native.ERR_TIMEOUT
    finally:
        g.set_option(native.OPT_FAULT_INJECT, 0)
        g.set_option(native.OPT_TIMEOUT_NS, 2_000_000_000)
    # The handle stays usable.
    C = g.run_mx(dA, dB, psa, psb, layout="TN")
    assert g.sync_status() == native.OK
    got = C.cpu().view(torch.int16).numpy().view(np.uint16)
    assert_exact(got, oracle.gemm_blockscaled(A, B, sa, sb, "TN", "e4m3", "bf16"), "after the timeout")


def test_invalid_arguments_and_k_zero(g):
    A = torch.zeros((32, 32)).to(torch.float8_e4m3fn).cuda()
    B = torch.zeros((32, 32)).to(torch.float8_e4m3fn).cuda()
    C = torch.zeros((32, 32), dtype=torch.bfloat16, device="cuda")
    s = g.pack_scales(torch.full((32, 1), 127, dtype=torch.uint8, device="cuda"), 32)
    a, b, c, p = A.data_ptr(), B.data_ptr(), C.data_ptr(), s.data_ptr()

    def mx(sfa=p, sfb=p, **kw):
        args = dict(M=32, N=32, K=32, lda=32, ldb=32, ldc=32, layout=0, dtype=native.DTYPE_E4M3,
                    out_dtype=native.DTYPE_BF16, alpha=1.0, beta=0.0)
        args.update(kw)
        return g.run_mx_raw(a, b, c, sfa, sfb, args["M"], args["N"], args["K"], args["lda"], args["ldb"],
                            args["ldc"], args["layout"], args["dtype"], args["out_dtype"], args["alpha"],
                            args["beta"])

    assert mx() == native.OK
    assert g.sync_status() == native.OK
    assert mx(dtype=native.DTYPE_BF16) == native.ERR_INVALID_ARG   # 16-bit operands take gemm_run_ex
    assert mx(sfa=0) == native.ERR_INVALID_ARG
    assert mx(sfb=0) == native.ERR_INVALID_ARG
    assert mx(sfa=p + 8) == native.ERR_UNSUPPORTED
    assert mx(out_dtype=native.DTYPE_E5M2) == native.ERR_INVALID_ARG
    # K == 0: C = beta * C, no scales needed.
    C.fill_(3.0)
    assert mx(sfa=0, sfb=0, K=0, beta=0.5) == native.OK
    assert g.sync_status() == native.OK
    assert torch.all(C == 1.5)
    # The packer validates its arguments.
    assert g._lib.gemm_mx_pack_scales(g._h, None, 4, 4, 4, p, None) == native.ERR_INVALID_ARG
    assert g._lib.gemm_mx_pack_scales(g._h, p, 4, 4, 3, p, None) == native.ERR_INVALID_ARG
    assert g._lib.gemm_mx_pack_scales(g._h, p, 0, 4, 4, p, None) == native.OK

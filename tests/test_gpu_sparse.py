"""GPU parity of 2:4 structured sparsity (gemm_sp_compress + gemm_run_sp) against the oracle.

The method of "张量缩并：mma 语法" (structured sparsity): A has at most two non-zeros in every
four consecutive elements along K; it is stored as the kept values plus metadata naming their
positions, and the sparse contraction multiplies each kept value by the B row it came from.
The result is the dense product of the 2:4 matrix, so the dense oracle is the reference;
the oracle's own compressor and sparse contraction check the compressed form.

Bar: integer operands in {-2..2} are bit-exact (every partial sum an integer below 2^24);
normal operands within atol = rtol = 1e-2 (fp16 C) / 3e-2 (bf16 C).
"""
import numpy as np
import pytest
import torch

from dense_tiled_gemm_04_gb300 import native
from dense_tiled_gemm_04_gb300.workloads import make_inputs, prune_24, round_up

import oracle
from test_gpu_fp8 import int_c
from test_gpu_parity import SENTINEL, assert_close, assert_exact, codes, to_device

pytestmark = pytest.mark.gpu

NAN16 = {"f16": 0x7E00, "bf16": 0x7FC0}
TDT = {"f16": torch.float16, "bf16": torch.bfloat16}


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


def unpack_meta(meta: np.ndarray, M: int, K: int) -> np.ndarray:
    """The chunked metadata written back as plain words (M x ceil(K/32)), from the layout's
    definition: chunk (rb, s) at (rb * S + s) * 4096, word 2s + h in half h (2048 bytes), lane
    l at l * 16; rows r = 16 b + i and r + 8 (i < 8) share lanes r (groups 0-3: row r in the
    low 16 bits, row r + 8 in the high) and r + 8 (groups 4-7, the same way).  Nibbles of
    groups past K are cleared (the oracle leaves them 0)."""
    S = -(-K // 64)
    words = meta.view(np.uint32)
    out = np.zeros((M, -(-K // 32)), np.uint32)
    for m in range(M):
        lane = m % 128
        lo_lane, hi_lane = (lane, lane + 8) if lane % 16 < 8 else (lane - 8, lane)
        shift = 0 if lane % 16 < 8 else 16
        for j in range(out.shape[1]):
            s, h = j // 2, j % 2
            base = ((m // 128) * S + s) * 1024 + h * 512
            lo = (int(words[base + lo_lane * 4]) >> shift) & 0xFFFF
            hi = (int(words[base + hi_lane * 4]) >> shift) & 0xFFFF
            out[m, j] = lo | (hi << 16)
    groups = K // 4
    for j in range(out.shape[1]):
        valid = min(8, groups - 8 * j)
        if valid < 8:
            out[:, j] &= np.uint32((1 << (4 * valid)) - 1)
    return out


def compress(g, A_cpu):
    dA = to_device(A_cpu)
    Ac, meta, bad = g.sp_compress(dA)
    torch.cuda.synchronize()
    return Ac, meta, int(bad.item())


def run_sp(g, Ac, meta, B, layout, dtype, alpha=1.0, beta=0.0, col_major=False, c_init=None, pad=8, extra=2):
    """gemm_run_sp with C in a sentinel-filled buffer.  Returns (logical M x N codes, guard ok)."""
    M, K = Ac.shape[0], 2 * Ac.shape[1]
    N = B.shape[1] if layout == "NN" else B.shape[0]
    rows, cols = (N, M) if col_major else (M, N)
    ldc = round_up(max(cols, 1), 8) + pad
    buf = torch.full((rows + extra, ldc), 0, dtype=torch.int16)
    buf.fill_(SENTINEL)
    window = buf[:rows, :cols]
    logical = window.t() if col_major else window
    if c_init is None:
        logical.fill_(NAN16[dtype] - 65536 if NAN16[dtype] > 32767 else NAN16[dtype])
    else:
        logical.copy_(torch.from_numpy(c_init.view(np.int16)))
    dbuf = buf.cuda()
    dB = to_device(B)
    lda = Ac.stride(0) if M > 1 else round_up(max(K // 2, 1), 8)
    ldb = dB.stride(0) if B.shape[0] > 1 else round_up(max(B.shape[1], 1), 8)
    st = g.run_sp_raw(Ac.data_ptr(), dB.data_ptr(), dbuf.data_ptr(), meta.data_ptr(), M, N, K, lda, ldb, ldc,
                      native.LAYOUTS[layout], native.DTYPES[dtype], alpha, beta, int(col_major), 0)
    assert st == native.OK, native.status_string(st)
    assert g.sync_status() == native.OK
    res = dbuf.cpu().numpy().view(np.uint16)
    win = res[:rows, :cols]
    guard = res.copy()
    guard[:rows, :cols] = SENTINEL
    return np.ascontiguousarray(win.T if col_major else win), bool(np.all(guard == SENTINEL))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("shape", [(300, 520), (129, 100), (1, 4), (256, 4096)])
def test_compress_matches_the_oracle(g, dtype, shape):
    M, K = shape
    A, _ = make_inputs(M, 8, K, "NN", dtype, "normal", seed=101)
    A = prune_24(A, seed=102)
    if M > 2 and K >= 8:
        A[1, 4:8] = torch.tensor([1.0, 2.0, 3.0, 0.0])  # one group with three non-zeros
        A[2, 0:4] = torch.tensor([-0.0, 0.0, 0.0, 5.0])  # negative zero counts as zero
    Ac, meta, bad = compress(g, A)
    ref_ac, ref_e, ref_bad = oracle.sparse24_compress(A)
    assert bad == ref_bad
    assert np.array_equal(codes(Ac), ref_ac)
    got_e = unpack_meta(meta.cpu().numpy(), M, K)
    assert np.array_equal(got_e, ref_e)
    assert meta.numel() >= native.sp_meta_bytes(M, K)


@pytest.mark.parametrize("config", CONFIGS, indirect=True)
@pytest.mark.parametrize("layout", ["NN", "TN"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_int_operands_bit_exact(g, config, layout, dtype):
    M, N, K = 300, 257, 520  # ragged M, N; K = 8 stages of 64 + 8
    A, B = make_inputs(M, N, K, layout, dtype, "int", seed=103)
    A = prune_24(A, seed=104)
    Ac, meta, bad = compress(g, A)
    assert bad == 0
    got, guard = run_sp(g, Ac, meta, B, layout, dtype)
    assert guard
    assert_exact(got, oracle.gemm(A, B, layout, dtype), f"{dtype} {layout}")


@pytest.mark.parametrize("layout", ["NN", "TN"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_normal_operands_within_tolerance(g, layout, dtype):
    M, N, K = 515, 389, 1000
    A, B = make_inputs(M, N, K, layout, dtype, "normal", seed=105, scale=1 / 16)
    A = prune_24(A, seed=106)
    Ac, meta, _ = compress(g, A)
    got, guard = run_sp(g, Ac, meta, B, layout, dtype)
    assert guard
    assert_close(got, oracle.gemm(A, B, layout, dtype), dtype, f"{dtype} {layout}")


@pytest.mark.parametrize("config", CONFIGS, indirect=True)
def test_one_kept_value_selects_its_b_row(g, config):
    # A single 1.0 at K position k of row m: row m of C is row k of B (NN), for positions in
    # every nibble of both metadata words of a stage and in a later stage, in both CTAs' rows
    # of a pair tile (256 rows).
    M, N, K = 256, 64, 192
    _, B = make_inputs(M, N, K, "NN", "f16", "int", seed=107)
    A = torch.zeros((M, K), dtype=torch.float16)
    picks = [(0, 0), (1, 1), (2, 6), (3, 7), (5, 13), (31, 31), (32, 33), (40, 62), (77, 63), (100, 64), (127, 191),
             (128, 2), (137, 11), (150, 40), (200, 127), (255, 190)]
    for m, k in picks:
        A[m, k] = 1.0
    Ac, meta, bad = compress(g, A)
    assert bad == 0
    got, _ = run_sp(g, Ac, meta, B, "NN", "f16")
    bc = codes(B)
    for m, k in picks:
        assert np.array_equal(got[m], bc[k]), (m, k)


@pytest.mark.parametrize("config", CONFIGS[1:], indirect=True)
@pytest.mark.parametrize("col_major", [False, True])
@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_accumulate_and_column_major_bit_exact(g, config, col_major, layout):
    M, N, K = 333, 200, 264
    A, B = make_inputs(M, N, K, layout, "bf16", "int", seed=108)
    A = prune_24(A, seed=109)
    Ac, meta, _ = compress(g, A)
    c0 = int_c(M, N, "bf16", seed=110)
    got, guard = run_sp(g, Ac, meta, B, layout, "bf16", alpha=2.0, beta=-0.5, col_major=col_major, c_init=c0)
    assert guard
    ref_ac, ref_e, _ = oracle.sparse24_compress(A)
    ref = oracle.gemm_sparse24(ref_ac, ref_e, B, layout, "bf16", alpha=2.0, beta=-0.5, Cin=c0)
    assert_exact(got, ref, f"{layout} col_major={col_major}")


@pytest.mark.parametrize("shape", [(1, 1, 4), (7, 9, 16), (128, 256, 64), (129, 257, 132), (64, 48, 40),
                                   (3, 600, 36), (200, 136, 4096)])
@pytest.mark.parametrize("config", CONFIGS[1:], indirect=True)
@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_edge_shapes(g, config, shape, layout):
    M, N, K = shape
    A, B = make_inputs(M, N, K, layout, "f16", "int", seed=111)
    A = prune_24(A, seed=112)
    Ac, meta, _ = compress(g, A)
    got, guard = run_sp(g, Ac, meta, B, layout, "f16")
    assert guard
    assert_exact(got, oracle.gemm(A, B, layout, "f16"), f"{shape} {layout}")


@pytest.mark.parametrize("config", CONFIGS[1:], indirect=True)
@pytest.mark.parametrize("stream_k,k_snake", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_multi_tile_stream_k_bit_exact(g, config, stream_k, k_snake):
    M, N, K = 16384, 1024, 2048
    A, B = make_inputs(M, N, K, "TN", "bf16", "int", seed=113)
    A = prune_24(A, seed=114)
    Ac, meta, _ = compress(g, A)
    snake0 = g.get_option(native.OPT_K_SNAKE)
    g.set_option(native.OPT_STREAM_K, stream_k)
    g.set_option(native.OPT_K_SNAKE, k_snake)
    try:
        C = g.run_sp(Ac, B.cuda(), meta, layout="TN")
        torch.cuda.synchronize()
        assert g.sync_status() == native.OK
    finally:
        g.set_option(native.OPT_STREAM_K, 1)
        g.set_option(native.OPT_K_SNAKE, snake0)
    assert_exact(codes(C), oracle.gemm(A, B, "TN", "bf16"), f"stream_k={stream_k} k_snake={k_snake}")


@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_full_size_8192_full_matrix(g, layout):
    M = N = K = 8192
    A, B = make_inputs(M, N, K, layout, "bf16", "normal", seed=116, scale=1 / 64)
    A = prune_24(A, seed=117)
    Ac, meta, bad = compress(g, A)
    assert bad == 0
    C = g.run_sp(Ac, B.cuda(), meta, layout=layout)
    torch.cuda.synchronize()
    assert g.sync_status() == native.OK
    assert_close(codes(C), oracle.gemm(A, B, layout, "bf16"), "bf16", f"8192^3 {layout}")


@pytest.mark.parametrize("config", CONFIGS[1:], indirect=True)
def test_watchdog_reports_a_timeout(g, config):
    M, N, K = 512, 512, 1024
    A, B = make_inputs(M, N, K, "TN", "f16", "int", seed=119)
    A = prune_24(A, seed=120)
    Ac, meta, _ = compress(g, A)
    dB = B.cuda()
    g.set_option(native.OPT_TIMEOUT_NS, 20_000_000)
    g.set_option(native.OPT_FAULT_INJECT, 1)
    try:
        g.run_sp(Ac, dB, meta, layout="TN")
        assert g.sync_status() == native.ERR_TIMEOUT
    finally:
        g.set_option(native.OPT_FAULT_INJECT, 0)
        g.set_option(native.OPT_TIMEOUT_NS, 2_000_000_000)
    C = g.run_sp(Ac, dB, meta, layout="TN")
    assert g.sync_status() == native.OK
    assert_exact(codes(C), oracle.gemm(A, B, "TN", "f16"), "after the timeout")


def test_invalid_arguments_and_k_zero(g):
    Ac = torch.zeros((32, 16), dtype=torch.float16, device="cuda")
    B = torch.zeros((32, 32), dtype=torch.float16, device="cuda")
    C = torch.zeros((32, 32), dtype=torch.float16, device="cuda")
    meta = torch.full((native.sp_meta_bytes(32, 32),), 0x44, dtype=torch.uint8, device="cuda")
    a, b, c, e = Ac.data_ptr(), B.data_ptr(), C.data_ptr(), meta.data_ptr()

    def sp(meta_ptr=e, **kw):
        args = dict(M=32, N=32, K=32, lda=16, ldb=32, ldc=32, layout=0, dtype=native.DTYPE_F16, alpha=1.0, beta=0.0)
        args.update(kw)
        return g.run_sp_raw(a, b, c, meta_ptr, args["M"], args["N"], args["K"], args["lda"], args["ldb"], args["ldc"],
                            args["layout"], args["dtype"], args["alpha"], args["beta"])

    assert sp() == native.OK
    assert g.sync_status() == native.OK
    assert sp(K=30, lda=16) == native.ERR_UNSUPPORTED   # K not a multiple of 4
    assert sp(lda=8) == native.ERR_INVALID_ARG          # lda < K / 2
    assert sp(meta_ptr=0) == native.ERR_INVALID_ARG
    assert sp(meta_ptr=e + 8) == native.ERR_UNSUPPORTED
    assert sp(dtype=native.DTYPE_E4M3) == native.ERR_INVALID_ARG
    C.fill_(2.0)
    assert sp(meta_ptr=0, K=0, beta=-1.0) == native.OK  # C = beta * C
    assert g.sync_status() == native.OK
    assert torch.all(C == -2.0)
    A = torch.zeros((4, 6), dtype=torch.float16, device="cuda")
    with pytest.raises(ValueError):
        g.sp_compress(A)

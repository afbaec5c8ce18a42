"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bar: bit-exact on integer-valued inputs (every partial sum is an integer of magnitude
<= 4K < 2^24, exact in fp32 in any order, then one round-to-nearest-even on both sides);
within |gpu - ref| <= atol + rtol*|ref| otherwise, with atol = rtol = 1e-2 for fp16
output and 3e-2 for bf16 output.  Every output element is compared, at every size up to
the full-size workloads (whose oracle results are computed once per input set and shared
by the tests that use them).
"""
import functools

import numpy as np
import pytest
import torch

from dense_tiled_gemm_04_gb300 import native
from dense_tiled_gemm_04_gb300.workloads import WORKLOADS, make_inputs, round_up, workload_inputs

import oracle

pytestmark = pytest.mark.gpu

TOL = {"f16": (1e-2, 1e-2), "bf16": (3e-2, 3e-2)}
SENTINEL = 0x7777  # a finite 16-bit code that C = A·B never produces in these tests


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


def to_device(x: torch.Tensor) -> torch.Tensor:
    """Copy a (possibly row-padded) CPU view to the GPU keeping its row pitch; a row pitch
    that is not a multiple of 8 elements is widened to one (NaN padding)."""
    rows, cols = x.shape
    if x.numel() == 0:
        return x.cuda()
    if rows > 1 and x.stride(0) % 8 != 0:
        buf = torch.full((rows, round_up(cols, 8)), float("nan"), dtype=x.dtype)
        buf[:, :cols] = x
        x = buf[:, :cols]
    ld = x.stride(0) if rows > 1 else cols
    base = x.as_strided((rows, ld), (ld, 1)) if rows > 1 else x
    return base.cuda()[:, :cols]


def codes(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def gpu_gemm(g, A, B, layout, dtype, extra_rows=0, ldc_pad=0, stream=None):
    """Run through the C ABI; C sits in a sentinel-filled buffer with spare rows/columns.

    Returns (C codes M x N, whole buffer codes) so callers can check the guard region."""
    M, K = A.shape
    N = B.shape[1] if layout == "NN" else B.shape[0]
    ldc = round_up(max(N, 1), 8) + ldc_pad
    tdt = A.dtype
    buf = torch.full((M + extra_rows, ldc), 0, dtype=torch.int16, device="cuda")
    buf.fill_(SENTINEL)
    buf = buf.view(tdt)
    C = buf[:M, :N]
    dA, dB = to_device(A), to_device(B)
    lda = dA.stride(0) if M > 1 else round_up(max(K, 1), 8)
    brows = B.shape[0]
    ldb = dB.stride(0) if brows > 1 else round_up(max(B.shape[1], 1), 8)
    s = 0 if stream is None else stream.cuda_stream
    st = g.run_raw(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, lda, ldb, ldc,
                   native.LAYOUTS[layout], native.DTYPES[dtype], s)
    assert st == native.OK, native.status_string(st)
    assert g.sync_status(stream) == native.OK
    return codes(C), codes(buf)


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what=""):
    a, r = oracle.decode(got, dtype), oracle.decode(ref, dtype)
    atol, rtol = TOL[dtype]
    bad = ~(np.abs(a - r) <= atol + rtol * np.abs(r))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first at {idx.tolist()}: "
                             f"gpu {a[tuple(idx[0])]} ref {r[tuple(idx[0])]}")


def assert_exact(got: np.ndarray, ref: np.ndarray, what=""):
    bad = got != ref
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} codes differ; first at {idx.tolist()}: "
                             f"gpu {got[tuple(idx[0])]:#06x} ref {ref[tuple(idx[0])]:#06x}")


def assert_guard(buf: np.ndarray, M: int, N: int):
    guard = buf.copy()
    guard[:M, :N] = SENTINEL
    assert np.all(guard == SENTINEL), "a write landed outside the M x N window of C"


# ------------------------------------------------------------------ the five workloads


@pytest.mark.parametrize("name", ["c1", "c2"])
@pytest.mark.parametrize("dist", ["workload", "int"])
def test_small_workloads_full(g, name, dist):
    w = WORKLOADS[name]
    if dist == "int":
        w = w.with_dist("int")
    A, B = workload_inputs(w)
    got, buf = gpu_gemm(g, A, B, w.layout, w.dtype, extra_rows=2, ldc_pad=8)
    ref = oracle.gemm(A, B, w.layout, w.dtype)
    assert_guard(buf, w.M, w.N)
    if dist == "int":
        assert_exact(got, ref, f"{name} int")
    else:
        assert_close(got, ref, w.dtype, name)


@functools.lru_cache(maxsize=2)
def workload_case(name: str, dist: str):
    """(workload, A, B, the oracle's C) for a workload with its own distribution ("workload")
    or integer inputs ("int"); the oracle runs once per input set."""
    w = WORKLOADS[name]
    if dist == "int":
        w = w.with_dist("int")
    A, B = workload_inputs(w)
    oracle.build()
    return w, A, B, oracle.gemm(A, B, w.layout, w.dtype)


@pytest.mark.parametrize("name", ["c3", "c4", "c5"])
@pytest.mark.parametrize("dist", ["workload", "int"])
def test_full_size_workloads_full_matrix(g, name, dist):
    # Every element of C against the oracle, under the library's own choice and both forced
    # configurations, with a guard row and guard columns around C.
    w, A, B, ref = workload_case(name, dist)
    for config in (native.CONFIG_AUTO, native.CONFIG_128x256, native.CONFIG_256x256):
        g.set_option(native.OPT_CONFIG, config)
        try:
            got, buf = gpu_gemm(g, A, B, w.layout, w.dtype, extra_rows=1, ldc_pad=8)
        finally:
            g.set_option(native.OPT_CONFIG, native.CONFIG_AUTO)
        assert_guard(buf, w.M, w.N)
        if dist == "int":
            assert_exact(got, ref, f"{name} int config {config}")
        else:
            assert_close(got, ref, w.dtype, f"{name} config {config}")


# ------------------------------------------------------------------ edges and pins

SHAPES = [(1, 1, 1), (1, 8, 3), (3, 5, 7), (8, 8, 8), (17, 9, 33), (64, 64, 64), (65, 97, 130),
          (127, 129, 63), (128, 256, 64), (129, 257, 65), (200, 300, 1), (255, 511, 200), (1, 1000, 129),
          (300, 1, 77), (257, 130, 1000)]


@pytest.mark.parametrize("layout", ["NN", "TN"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("config", [native.CONFIG_128x256, native.CONFIG_128x128, native.CONFIG_128x64,
                                    native.CONFIG_256x256])
def test_ragged_shapes(g, layout, dtype, config):
    g.set_option(native.OPT_CONFIG, config)
    try:
        for i, (M, N, K) in enumerate(SHAPES):
            for dist in ("int", "normal"):
                bcols = N if layout == "NN" else K
                A, B = make_inputs(M, N, K, layout, dtype, dist, seed=1000 + i,
                                   lda=round_up(K, 8) + (8 if i % 2 else 0),
                                   ldb=round_up(bcols, 8) + (8 if i % 3 == 0 else 0))
                got, buf = gpu_gemm(g, A, B, layout, dtype, extra_rows=1, ldc_pad=8 * (i % 2))
                ref = oracle.gemm(A, B, layout, dtype)
                assert_guard(buf, M, N)
                what = f"{(M, N, K)} {layout} {dtype} {dist} cfg{config}"
                if dist == "int":
                    assert_exact(got, ref, what)
                else:
                    assert_close(got, ref, dtype, what)
    finally:
        g.set_option(native.OPT_CONFIG, native.CONFIG_AUTO)


@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_tail_all_ones_is_130(g, layout):
    # M=65, N=97, K=130: leading dimensions padded to multiples of 8 (136, 104) while the
    # logical sizes stay ragged; every output must be 130, not 128.
    M, N, K = 65, 97, 130
    A, B = make_inputs(M, N, K, layout, "f16", "ones", seed=0, lda=136, ldb=104 if layout == "NN" else 136)
    got, buf = gpu_gemm(g, A, B, layout, "f16", extra_rows=3, ldc_pad=8)
    vals = oracle.decode(got, "f16")
    assert np.all(vals == 130.0), np.unique(vals)
    assert_guard(buf, M, N)


def test_fp32_accumulation_pin(g):
    # Row [2048, 1, 1] times column [1, 1, 1]: 2050 only if partial sums are kept in fp32.
    A = torch.tensor([[2048.0, 1.0, 1.0]], dtype=torch.float16)
    B = torch.ones((3, 1), dtype=torch.float16)
    got, _ = gpu_gemm(g, A, B, "NN", "f16")
    assert oracle.decode(got, "f16")[0, 0] == 2050.0
    # Same in the TN layout and with the 1s spread across two K blocks of 64.
    A2 = torch.zeros((1, 130), dtype=torch.float16)
    A2[0, 0], A2[0, 64], A2[0, 129] = 2048.0, 1.0, 1.0
    B2 = torch.ones((1, 130), dtype=torch.float16)
    got2, _ = gpu_gemm(g, A2, B2, "TN", "f16")
    assert oracle.decode(got2, "f16")[0, 0] == 2050.0


@pytest.mark.parametrize("layout", ["NN", "TN"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_identity_and_permutation(g, layout, dtype):
    M, K = 300, 384
    A, _ = make_inputs(M, K, K, layout, dtype, "uniform", seed=77)
    eye = torch.eye(K, dtype=A.dtype)
    got, _ = gpu_gemm(g, A, eye, layout, dtype)
    assert_exact(got, oracle._codes(A), "A·I")
    perm = torch.randperm(K, generator=torch.Generator().manual_seed(3))
    P = torch.zeros(K, K, dtype=A.dtype)
    P[perm, torch.arange(K)] = 1
    got, _ = gpu_gemm(g, A, P if layout == "NN" else P.T.contiguous(), layout, dtype)
    assert_exact(got, oracle._codes(A)[:, perm.numpy()], "A·P")


def test_k_zero_writes_zeros_and_m_n_zero_is_noop(g):
    for dtype in ("f16", "bf16"):
        A = torch.empty((37, 0), dtype=native_dtype(dtype))
        B = torch.empty((0, 45), dtype=native_dtype(dtype))
        got, buf = gpu_gemm(g, A, B, "NN", dtype, extra_rows=1, ldc_pad=8)
        assert np.all(got == 0)
        assert_guard(buf, 37, 45)
    C = torch.full((4, 8), 3.0, dtype=torch.float16, device="cuda")
    for (M, N) in [(0, 8), (4, 0)]:
        st = g.run_raw(C.data_ptr(), C.data_ptr(), C.data_ptr(), M, N, 8, 8, 8, 8, 0, 0, 0)
        assert st == native.OK
    torch.cuda.synchronize()
    assert torch.all(C == 3.0)


def native_dtype(dtype):
    return {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]


@pytest.mark.parametrize("config", [native.CONFIG_AUTO, native.CONFIG_256x256])
@pytest.mark.parametrize("layout", ["TN", "NN"])
def test_several_tiles_per_cta_and_raster_groups(g, config, layout):
    M, N, K = 1000, 1000, 520
    A, B = make_inputs(M, N, K, layout, "f16", "int", seed=5)
    ref = oracle.gemm(A, B, layout, "f16")
    g.set_option(native.OPT_CONFIG, config)
    try:
        for max_ctas, group in [(1, 16), (3, 1), (7, 3), (0, 64), (5, 1000), (2, 2)]:
            g.set_option(native.OPT_MAX_CTAS, max_ctas)
            g.set_option(native.OPT_RASTER_GROUP, group)
            got, _ = gpu_gemm(g, A, B, layout, "f16")
            assert_exact(got, ref, f"cfg{config} max_ctas={max_ctas} group={group}")
    finally:
        g.set_option(native.OPT_MAX_CTAS, 0)
        g.set_option(native.OPT_RASTER_GROUP, 0)
        g.set_option(native.OPT_CONFIG, native.CONFIG_AUTO)


def test_plan_kind_reports_the_launch_of_each_operand_kind(g):
    # What gemm_run_sp / gemm_run_mx launch for 8192^3 TN by default: the CTA pair (7-stage
    # ring, 7 warps) for a 2:4-sparse A, the CTA pair (6 stages, 7 warps) for block scales; a
    # small block-scaled problem takes the one-CTA 128 x 256 tile (4 stages).
    sp = g.plan(8192, 8192, 8192, "TN", "bf16", "sparse24")
    assert (sp["config"], sp["cluster"], sp["bm"], sp["bn"], sp["stages"], sp["threads"]) == \
        (native.CONFIG_256x256, 2, 256, 256, 7, 224)
    mx = g.plan(8192, 8192, 8192, "TN", "e4m3", "block_scaled")
    assert (mx["config"], mx["cluster"], mx["bm"], mx["bn"], mx["stages"], mx["threads"]) == \
        (native.CONFIG_256x256, 2, 256, 256, 6, 224)
    small = g.plan(1000, 1000, 1000, "TN", "e4m3", "block_scaled")
    assert (small["config"], small["cluster"], small["bn"], small["stages"], small["threads"]) == \
        (native.CONFIG_128x256, 1, 256, 4, 224)
    assert g.plan(8192, 8192, 8192, "TN", "bf16")["threads"] == 192
    assert g.plan(8192, 8192, 8192, "TN", "bf16") == g.plan(8192, 8192, 8192, "TN", "bf16", "dense")
    for dtype, kind in (("bf16", "block_scaled"), ("e4m3", "sparse24")):
        with pytest.raises(native.GemmError):
            g.plan(64, 64, 64, "TN", dtype, kind)


def test_host_chunk_options_defaults_and_limits(g):
    assert g.get_option(native.OPT_HOST_ROW_CHUNKS) == 8
    assert g.get_option(native.OPT_HOST_COL_CHUNKS) == 4
    for opt, hi in ((native.OPT_HOST_ROW_CHUNKS, 16), (native.OPT_HOST_COL_CHUNKS, 8)):
        for bad in (0, hi + 1):
            with pytest.raises(native.GemmError):
                g.set_option(opt, bad)
    assert g.get_option(native.OPT_HOST_ROW_CHUNKS) == 8


def test_k_snake_option_default_limits_and_plan(g):
    assert g.get_option(native.OPT_K_SNAKE) == 1
    for bad in (-1, 2):
        with pytest.raises(native.GemmError):
            g.set_option(native.OPT_K_SNAKE, bad)
    assert g.get_option(native.OPT_K_SNAKE) == 1
    # The plan reports the K order the launch uses: block-scaled kernels always walk forward.
    assert g.plan(8192, 8192, 8192, "TN", "bf16")["k_snake"] == 1
    assert g.plan(8192, 8192, 8192, "TN", "e4m3")["k_snake"] == 1
    assert g.plan(8192, 8192, 8192, "TN", "bf16", "sparse24")["k_snake"] == 1
    assert g.plan(8192, 8192, 8192, "TN", "e4m3", "block_scaled")["k_snake"] == 0
    g.set_option(native.OPT_K_SNAKE, 0)
    try:
        assert g.plan(8192, 8192, 8192, "TN", "bf16")["k_snake"] == 0
    finally:
        g.set_option(native.OPT_K_SNAKE, 1)


def test_plan_reports_pair_clusters(g):
    g.set_option(native.OPT_CONFIG, native.CONFIG_256x256)
    try:
        pl = g.plan(8192, 8192, 8192, "TN", "bf16")
    finally:
        g.set_option(native.OPT_CONFIG, native.CONFIG_AUTO)
    assert pl["cluster"] == 2 and pl["bm"] == 256 and pl["bn"] == 256
    assert pl["grid"] % 2 == 0 and 2 <= pl["grid"] <= torch.cuda.get_device_properties(0).multi_processor_count
    assert pl["tiles_m"] == 32 and pl["tiles_n"] == 32 and pl["k_blocks"] == 128


def test_automatic_raster_group_follows_the_a_panel_bytes(g):
    # The tile rows whose A holds about 48 MiB, at most 16 and at most the tile columns: 12 rows
    # of 256 x 8192 bf16 (4 MiB each), 16 of E4M3 or of a 2:4-compressed bf16 A (2 MiB each,
    # 24 capped), 4 on the 4-column tall-skinny grid; an explicit option wins.
    assert g.plan(8192, 8192, 8192, "TN", "bf16")["raster_group"] == 12
    assert g.plan(4096, 4096, 4096, "NN", "f16")["raster_group"] == 16
    assert g.plan(8192, 8192, 8192, "TN", "e4m3")["raster_group"] == 16
    assert g.plan(8192, 8192, 8192, "TN", "e4m3", "block_scaled")["raster_group"] == 16
    assert g.plan(8192, 8192, 8192, "TN", "bf16", "sparse24")["raster_group"] == 16
    assert g.plan(16384, 1024, 8192, "TN", "f16")["raster_group"] == 4
    assert g.plan(128, 256, 192, "NN", "f16")["raster_group"] == 4  # 4 tiles of 128 x 64
    g.set_option(native.OPT_RASTER_GROUP, 3)
    try:
        assert g.plan(16384, 1024, 8192, "TN", "f16")["raster_group"] == 3
    finally:
        g.set_option(native.OPT_RASTER_GROUP, 0)


def test_plan_of_the_narrow_tile(g):
    # 128 x 64 on one CTA, 8-stage ring, for 16-bit dense operands; 8-bit operands take
    # 128 x 128 (an N-major 8-bit B row is 128 wide), side-data kernels 128 x 256.
    g.set_option(native.OPT_CONFIG, native.CONFIG_128x64)
    try:
        pl = g.plan(1000, 1000, 1000, "NN", "f16")
        f8 = g.plan(1000, 1000, 1000, "NN", "e4m3")
        mx = g.plan(1000, 1000, 1024, "TN", "e4m3", "block_scaled")
        sp = g.plan(1000, 1000, 1000, "TN", "bf16", "sparse24")
    finally:
        g.set_option(native.OPT_CONFIG, native.CONFIG_AUTO)
    assert (pl["config"], pl["bm"], pl["bn"], pl["cluster"], pl["stages"]) == (native.CONFIG_128x64, 128, 64, 1, 8)
    assert pl["tiles_m"] == 8 and pl["tiles_n"] == 16
    assert (f8["config"], f8["bn"]) == (native.CONFIG_128x128, 128)
    for other in (mx, sp):
        assert (other["config"], other["bn"]) == (native.CONFIG_128x256, 256)


def test_large_extents(g):
    # Long M (131072 rows) and long N (65536 columns) with a short K: the TMA coordinates
    # and the tile scheduler at sizes far beyond the workloads' tile counts.
    for (M, N, K, layout) in [(131072, 136, 72, "TN"), (136, 65536, 72, "NN")]:
        A, B = make_inputs(M, N, K, layout, "bf16", "int", seed=M + N)
        got, _ = gpu_gemm(g, A, B, layout, "bf16")
        assert_exact(got, oracle.gemm(A, B, layout, "bf16"), f"{(M, N, K)}")


def test_side_stream(g):
    w = WORKLOADS["c2"].with_dist("int")
    A, B = workload_inputs(w)
    s = torch.cuda.Stream()
    got, _ = gpu_gemm(g, A, B, w.layout, w.dtype, stream=s)
    assert_exact(got, oracle.gemm(A, B, w.layout, w.dtype), "side stream")


def test_torch_binding_matmul(g):
    A, B = make_inputs(333, 444, 555, "NN", "bf16", "int", seed=8, lda=560, ldb=448)
    C = native.matmul(to_device(A), to_device(B), "NN")
    torch.cuda.synchronize()
    assert_exact(codes(C), oracle.gemm(A, B, "NN", "bf16"), "matmul")


def test_misaligned_arguments_are_rejected(g):
    A = torch.zeros((64, 72), dtype=torch.float16, device="cuda")
    B = torch.zeros((72, 64), dtype=torch.float16, device="cuda")
    C = torch.zeros((64, 72), dtype=torch.float16, device="cuda")
    ok = g.run_raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), 64, 64, 64, 72, 64, 72, 0, 0, 0)
    assert ok == native.OK
    assert g.run_raw(A.data_ptr() + 2, B.data_ptr(), C.data_ptr(), 64, 64, 64, 72, 64, 72, 0, 0, 0) \
        == native.ERR_UNSUPPORTED
    assert g.run_raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), 64, 64, 64, 68, 64, 72, 0, 0, 0) \
        == native.ERR_UNSUPPORTED
    assert g.run_raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), 64, 64, 64, 72, 64, 32, 0, 0, 0) \
        == native.ERR_INVALID_ARG
    assert g.sync_status() == native.OK


def test_run_host_matches_oracle(g):
    w = WORKLOADS["c2"]
    A, B = workload_inputs(w)
    C = torch.empty((w.M, w.N), dtype=A.dtype).pin_memory()
    st = g.run_host(A.pin_memory(), B.pin_memory(), C, w.layout)
    assert st == native.OK, native.status_string(st)
    assert_close(codes(C), oracle.gemm(A, B, w.layout, w.dtype), w.dtype, "run_host")


@pytest.mark.parametrize("layout", ["NN", "TN"])
@pytest.mark.parametrize("M,N,K,chunks", [(5000, 1000, 520, None), (4500, 4100, 264, None),
                                          (4500, 4100, 264, (1, 1)), (3000, 5000, 136, (16, 8))])
def test_run_host_pipelined_chunks_and_padding(g, layout, M, N, K, chunks):
    # The host path cuts A into row chunks and C's columns into column chunks (by default at
    # most 8 x 4, at least 1024 rows and 2048 columns: 5000 rows -> 4 x 1024 + 904; 4100
    # columns -> 2048 + 2048 + 4), and computes each block of C in its own launch as its
    # inputs arrive; host buffers have padded rows whose padding must be left alone (pitches
    # are multiples of 8 elements, as gemm_run_host requires).
    pad8 = lambda x: -(-x // 8) * 8  # noqa: E731
    A, B = make_inputs(M, N, K, layout, "bf16", "int", seed=12, lda=pad8(K + 8),
                       ldb=pad8((N if layout == "NN" else K) + 16))
    Ah = A.as_strided((M, A.stride(0)), (A.stride(0), 1)).pin_memory()[:, :K]
    rows_b = B.shape[0]
    Bh = B.as_strided((rows_b, B.stride(0)), (B.stride(0), 1)).pin_memory()[:, :B.shape[1]]
    ldc = pad8(N + 24)
    Cbuf = torch.full((M, ldc), 0, dtype=torch.int16).view(torch.bfloat16).pin_memory()
    Cbuf.view(torch.int16).fill_(SENTINEL)
    C = Cbuf[:, :N]
    try:
        if chunks is not None:
            g.set_option(native.OPT_HOST_ROW_CHUNKS, chunks[0])
            g.set_option(native.OPT_HOST_COL_CHUNKS, chunks[1])
        st = g.run_host(Ah, Bh, C, layout)
    finally:
        g.set_option(native.OPT_HOST_ROW_CHUNKS, 8)
        g.set_option(native.OPT_HOST_COL_CHUNKS, 4)
    assert st == native.OK, native.status_string(st)
    got = Cbuf.view(torch.int16).numpy().view(np.uint16)
    assert_guard(got, M, N)
    assert_exact(got[:, :N], oracle.gemm(A, B, layout, "bf16"), "run_host chunks")


@pytest.mark.parametrize("config", [native.CONFIG_AUTO, native.CONFIG_256x256])
def test_watchdog_timeout_is_reported_and_context_survives(g, config):
    # One ring stage is left unloaded and unarmed in the first unit: the MMA thread's wait on it must run out,
    # the kernel must leave cleanly, and the host must read GEMM_ERR_TIMEOUT.
    w = WORKLOADS["c2"].with_dist("int")
    A, B = workload_inputs(w)
    g.set_option(native.OPT_CONFIG, config)
    g.set_option(native.OPT_TIMEOUT_NS, 50_000_000)
    g.set_option(native.OPT_FAULT_INJECT, 1)
    try:
        dA, dB = to_device(A), to_device(B)
        C = native.empty_output(w.M, w.N, A.dtype, "cuda")
        st = g.run_raw(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), w.M, w.N, w.K, dA.stride(0), dB.stride(0),
                       C.stride(0), native.LAYOUTS[w.layout], native.DTYPES[w.dtype], 0)
        assert st == native.OK
        assert g.sync_status() == native.ERR_TIMEOUT
        info = g.error_info()
        # A timeout, first seen in the first CTA (or, for CTA pairs, either CTA of the first pair).
        first = {native.CONFIG_256x256: (0, 1)}.get(config, (0,))
        assert info[0] == 1 and info[2] in first, info
    finally:
        g.set_option(native.OPT_FAULT_INJECT, 0)
        g.set_option(native.OPT_TIMEOUT_NS, 2_000_000_000)
    # The context is still usable and the next run is correct.
    try:
        got, _ = gpu_gemm(g, A, B, w.layout, w.dtype)
    finally:
        g.set_option(native.OPT_CONFIG, native.CONFIG_AUTO)
    assert_exact(got, oracle.gemm(A, B, w.layout, w.dtype), "after timeout")


@pytest.mark.parametrize("config", [native.CONFIG_AUTO, native.CONFIG_128x128, native.CONFIG_128x64,
                                    native.CONFIG_256x256])
def test_dependent_gemms_on_one_stream(g, config):
    # GEMM launches may be scheduled while the stream's previous kernel drains; they must still
    # read that kernel's results.  Chain on one stream, no host sync in between: a torch kernel
    # rewrites A in place, C1 = A·B, C2 = C1·B2 (reads C1 as its A), then torch negates C2.
    M, N, K, N2 = 640, 512, 384, 256
    A, B = make_inputs(M, N, K, "NN", "f16", "int", seed=201)
    _, B2 = make_inputs(M, N2, N, "NN", "f16", "int", seed=202)
    dA, dB, dB2 = A.cuda(), B.cuda(), B2.cuda()
    g.set_option(native.OPT_CONFIG, config)
    try:
        for i in range(3):
            dA.copy_(A.cuda())
            dA.mul_(-1)                              # in-place torch kernel just before the GEMM
            C1 = g.run(dA, dB, layout="NN")
            C2 = g.run(C1, dB2, layout="NN")         # reads the previous GEMM's output
            C2.neg_()                                # in-place torch kernel just after
        torch.cuda.synchronize()
        assert g.sync_status() == native.OK
    finally:
        g.set_option(native.OPT_CONFIG, native.CONFIG_AUTO)
    negA = (-A.float()).to(torch.float16)
    ref1 = oracle.gemm(negA, B, "NN", "f16")
    assert_exact(codes(C1), ref1, "C1 = (-A)·B")
    c1_host = torch.from_numpy(ref1.view(np.int16)).view(torch.float16)
    ref2 = oracle.gemm(c1_host, B2, "NN", "f16")
    got2 = -oracle.decode(codes(C2), "f16")
    assert np.array_equal(got2, oracle.decode(ref2, "f16")), "C2 = C1·B2 read a stale C1"

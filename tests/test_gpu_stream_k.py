"""GPU parity of the stream-K schedule (the K blocks of the last tiles shared between CTAs).

Small CTA caps force many split tiles on shapes the oracle finishes quickly; integer
inputs must stay bit-exact, random inputs within tolerance, and a split run must give
the same bits every time (partial sums are merged in K order, whoever arrives last).
"""
import numpy as np
import pytest
import torch

from dense_tiled_gemm_04_gb300 import native
from dense_tiled_gemm_04_gb300.workloads import WORKLOADS, make_inputs, round_up

import oracle
from test_gpu_parity import assert_close, assert_exact, assert_guard, gpu_gemm, workload_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_tiled_gemm_04_gb300 import build

    build.build()
    oracle.build()
    h = native.Gemm(0)
    h.default_k_snake = h.get_option(native.OPT_K_SNAKE)
    yield h
    h.close()


def _with(g, **opts):
    names = {"config": native.OPT_CONFIG, "max_ctas": native.OPT_MAX_CTAS, "stream_k": native.OPT_STREAM_K,
             "group": native.OPT_RASTER_GROUP, "min_blocks": native.OPT_SK_MIN_BLOCKS,
             "split": native.OPT_SPLIT_MIN_BLOCKS, "k_snake": native.OPT_K_SNAKE}
    for k, v in opts.items():
        g.set_option(names[k], v)


def _reset(g):
    _with(g, config=native.CONFIG_AUTO, max_ctas=0, stream_k=1, group=0, min_blocks=8, split=32,
          k_snake=g.default_k_snake)


CASES = [
    # (M, N, K, layout, dtype, config, max_ctas)
    (1000, 1000, 2048, "TN", "f16", native.CONFIG_128x128, 24),
    (1000, 1000, 2048, "NN", "bf16", native.CONFIG_128x128, 10),
    (777, 1333, 1500, "NN", "f16", native.CONFIG_128x256, 8),
    (777, 1333, 1500, "TN", "bf16", native.CONFIG_128x256, 5),
    (1100, 1000, 1800, "TN", "f16", native.CONFIG_256x256, 12),
    (1100, 1000, 1800, "NN", "bf16", native.CONFIG_256x256, 6),
    (2000, 700, 3000, "TN", "bf16", native.CONFIG_256x256, 14),
    (1000, 1000, 2048, "TN", "bf16", native.CONFIG_128x64, 20),
    (1000, 1000, 2048, "NN", "f16", native.CONFIG_128x64, 7),
]


@pytest.mark.parametrize("case", CASES)
def test_stream_k_parity_and_plan(g, case):
    M, N, K, layout, dtype, config, max_ctas = case
    try:
        _with(g, config=config, max_ctas=max_ctas, stream_k=1)
        pl = g.plan(M, N, K, layout, dtype)
        tiles = pl["tiles_m"] * pl["tiles_n"]
        assert pl["dp_tiles"] < tiles, f"stream-K not engaged: {pl}"
        units = pl["grid"] // pl["cluster"]
        assert pl["sk_base"] * units + pl["sk_extra"] == (tiles - pl["dp_tiles"]) * pl["k_blocks"]
        for dist in ("int", "normal"):
            bcols = N if layout == "NN" else K
            A, B = make_inputs(M, N, K, layout, dtype, dist, seed=M + N + K,
                               lda=round_up(K, 8), ldb=round_up(bcols, 8))
            got, buf = gpu_gemm(g, A, B, layout, dtype, extra_rows=1, ldc_pad=8)
            assert_guard(buf, M, N)
            ref = oracle.gemm(A, B, layout, dtype)
            if dist == "int":
                assert_exact(got, ref, f"{case} int")
            else:
                assert_close(got, ref, dtype, f"{case} normal")
                again, _ = gpu_gemm(g, A, B, layout, dtype, extra_rows=1, ldc_pad=8)
                assert np.array_equal(got, again), "stream-K result changed between runs"
    finally:
        _reset(g)


@pytest.mark.parametrize("config", [native.CONFIG_128x128, native.CONFIG_256x256])
def test_stream_k_on_equals_off_on_integers(g, config):
    M, N, K = 1000, 1000, 2048
    A, B = make_inputs(M, N, K, "TN", "bf16", "int", seed=99)
    try:
        _with(g, config=config, max_ctas=12, stream_k=0)
        off, _ = gpu_gemm(g, A, B, "TN", "bf16")
        assert g.plan(M, N, K, "TN", "bf16")["dp_tiles"] == g.plan(M, N, K, "TN", "bf16")["tiles_m"] * \
            g.plan(M, N, K, "TN", "bf16")["tiles_n"]
        _with(g, stream_k=1)
        on, _ = gpu_gemm(g, A, B, "TN", "bf16")
    finally:
        _reset(g)
    assert_exact(on, off, "stream-K on vs off")


@pytest.mark.parametrize("name", ["c3", "c5"])
def test_default_plan_uses_stream_k_on_the_partial_wave_workloads(g, name):
    # 256 pair tiles on the pairs that fit at once leave a part-empty last wave.
    w = WORKLOADS[name]
    pl = g.plan(w.M, w.N, w.K, w.layout, w.dtype)
    tiles = pl["tiles_m"] * pl["tiles_n"]
    units = pl["grid"] // pl["cluster"]
    if tiles % units == 0:
        pytest.skip(f"{tiles} tiles fill {units} units exactly")
    assert pl["dp_tiles"] < tiles
    _, A, B, ref = workload_case(name, "int")
    got, _ = gpu_gemm(g, A, B, w.layout, w.dtype)
    assert_exact(got, ref, f"{name} int, default plan")


def test_c2_default_plan_fills_the_gpu_with_narrow_tiles(g):
    # 1000^3: 64 tiles of 128 x 128 would leave most SMs idle; the default plan runs 128 whole
    # tiles of 128 x 64 (16 K blocks each) on 128 CTAs.
    w = WORKLOADS["c2"]
    pl = g.plan(w.M, w.N, w.K, w.layout, w.dtype)
    assert (pl["config"], pl["bm"], pl["bn"]) == (native.CONFIG_128x64, 128, 64)
    assert pl["tiles_m"] * pl["tiles_n"] == 128 and pl["k_blocks"] == 16
    assert pl["grid"] == 128 and pl["dp_tiles"] == 128 and pl["sk_base"] == 0
    for dist in ("int", "normal"):
        A, B = make_inputs(w.M, w.N, w.K, w.layout, w.dtype, dist, seed=w.seed)
        got, buf = gpu_gemm(g, A, B, w.layout, w.dtype, extra_rows=1, ldc_pad=8)
        assert_guard(buf, w.M, w.N)
        ref = oracle.gemm(A, B, w.layout, w.dtype)
        if dist == "int":
            assert_exact(got, ref, "c2 int")
        else:
            assert_close(got, ref, w.dtype, "c2 normal")


@pytest.mark.parametrize("layout,dtype", [("TN", "f16"), ("NN", "bf16")])
def test_under_one_wave_split_when_shares_are_long(g, layout, dtype):
    # 1000 x 1000 x 8192: 64 tiles of 128 x 128 with 128 K blocks each, under one wave of 152
    # CTAs; shares of ~54 K blocks are long enough for the merge to pay, so every CTA works.
    # Forced 8-block shares on 128 x 128 tiles split 1000^3 over 128 CTAs (two shares per tile).
    M, N = 1000, 1000
    try:
        for K, opts, grid, base in ((8192, {}, 152, 53), (1000, dict(config=native.CONFIG_128x128, split=8), 128, 8)):
            _with(g, **opts)
            pl = g.plan(M, N, K, layout, dtype)
            units = pl["grid"] // pl["cluster"]
            assert pl["bn"] == 128 and pl["dp_tiles"] == 0 and pl["sk_base"] == base and pl["grid"] == grid, pl
            assert units > pl["tiles_m"] * pl["tiles_n"]
            for dist in ("int", "normal"):
                A, B = make_inputs(M, N, K, layout, dtype, dist, seed=K + len(opts))
                got, buf = gpu_gemm(g, A, B, layout, dtype, extra_rows=1, ldc_pad=8)
                assert_guard(buf, M, N)
                ref = oracle.gemm(A, B, layout, dtype)
                if dist == "int":
                    assert_exact(got, ref, f"K={K} int")
                else:
                    assert_close(got, ref, dtype, f"K={K} normal")
                    again, _ = gpu_gemm(g, A, B, layout, dtype, extra_rows=1, ldc_pad=8)
                    assert np.array_equal(got, again), "split result changed between runs"
            _reset(g)
    finally:
        _reset(g)


@pytest.mark.parametrize("min_blocks,grid", [(1, 6), (2, 2), (3, 2)])
@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_worked_example_split_by_shorter_shares(g, min_blocks, grid, layout):
    # 128 x 256 x 192 on 128 x 128 tiles: 2 tiles of 3 K blocks.  With shares of one K block
    # the two tiles run on 6 CTAs (three shares each); shares of two would give 3 CTAs, fewer
    # than two shares a tile, and shares of three one a tile: whole tiles on 2 CTAs.
    M, N, K = 128, 256, 192
    try:
        _with(g, config=native.CONFIG_128x128, split=min_blocks)
        pl = g.plan(M, N, K, layout, "f16")
        assert pl["grid"] == grid and pl["k_blocks"] == 3
        assert (pl["dp_tiles"] == 2) == (grid == 2)
        for dist in ("int", "uniform"):
            A, B = make_inputs(M, N, K, layout, "f16", dist, seed=0)
            got, buf = gpu_gemm(g, A, B, layout, "f16", extra_rows=1, ldc_pad=8)
            assert_guard(buf, M, N)
            ref = oracle.gemm(A, B, layout, "f16")
            if dist == "int":
                assert_exact(got, ref, f"min_blocks={min_blocks} int")
            else:
                assert_close(got, ref, "f16", f"min_blocks={min_blocks} uniform")
    finally:
        _reset(g)


@pytest.mark.parametrize("stream_k", [0, 1])
@pytest.mark.parametrize("case", CASES)
def test_k_snake_parity(g, case, stream_k):
    # Every second work item of a unit walks its K blocks from the last down.  The CTA caps
    # give each unit several whole tiles and (with stream-K) shares, so both directions run
    # on whole tiles and on shares merged through the workspace.
    M, N, K, layout, dtype, config, max_ctas = case
    try:
        _with(g, config=config, max_ctas=max_ctas, stream_k=stream_k, k_snake=1)
        pl = g.plan(M, N, K, layout, dtype)
        assert pl["tiles_m"] * pl["tiles_n"] > pl["grid"] // pl["cluster"]
        for dist in ("int", "normal"):
            bcols = N if layout == "NN" else K
            A, B = make_inputs(M, N, K, layout, dtype, dist, seed=M + N + K + 1,
                               lda=round_up(K, 8), ldb=round_up(bcols, 8))
            got, buf = gpu_gemm(g, A, B, layout, dtype, extra_rows=1, ldc_pad=8)
            assert_guard(buf, M, N)
            ref = oracle.gemm(A, B, layout, dtype)
            if dist == "int":
                assert_exact(got, ref, f"{case} int, k_snake")
            else:
                assert_close(got, ref, dtype, f"{case} normal, k_snake")
                again, _ = gpu_gemm(g, A, B, layout, dtype, extra_rows=1, ldc_pad=8)
                assert np.array_equal(got, again), "k_snake result changed between runs"
    finally:
        _reset(g)


@pytest.mark.parametrize("k_snake", [0, 1])
def test_k_snake_on_the_square_workload_int(g, k_snake):
    # The 8192^3 bf16 TN workload on its default plan (the CTA pair, 12 tile rows per group),
    # both K orders, every element against the oracle.
    w = WORKLOADS["c4"]
    _, A, B, ref = workload_case("c4", "int")
    try:
        _with(g, k_snake=k_snake)
        got, _ = gpu_gemm(g, A, B, w.layout, w.dtype)
    finally:
        _reset(g)
    assert_exact(got, ref, f"c4 int, k_snake={k_snake}")

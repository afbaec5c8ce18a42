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
    yield h
    h.close()


def _with(g, **opts):
    names = {"config": native.OPT_CONFIG, "max_ctas": native.OPT_MAX_CTAS, "stream_k": native.OPT_STREAM_K,
             "group": native.OPT_RASTER_GROUP}
    for k, v in opts.items():
        g.set_option(names[k], v)


def _reset(g):
    _with(g, config=native.CONFIG_AUTO, max_ctas=0, stream_k=1, group=16)


CASES = [
    # (M, N, K, layout, dtype, config, max_ctas)
    (1000, 1000, 2048, "TN", "f16", native.CONFIG_128x128, 24),
    (1000, 1000, 2048, "NN", "bf16", native.CONFIG_128x128, 10),
    (777, 1333, 1500, "NN", "f16", native.CONFIG_128x256, 8),
    (777, 1333, 1500, "TN", "bf16", native.CONFIG_128x256, 5),
    (1100, 1000, 1800, "TN", "f16", native.CONFIG_256x256, 12),
    (1100, 1000, 1800, "NN", "bf16", native.CONFIG_256x256, 6),
    (2000, 700, 3000, "TN", "bf16", native.CONFIG_256x256, 14),
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

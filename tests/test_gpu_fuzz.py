"""Seeded random sweep of shapes and launch options against the oracle (GPU).

Each case draws M, N, K (log-uniform, ragged), the layout, the 16-bit type, the kernel
configuration, stream-K on or off, the raster group, the K order of every second work item
and a cap on the number of CTAs, then runs integer-valued inputs through the C ABI and
compares with the oracle bit for bit, with sentinel guard rows and columns around C.  The epilogue sweep adds alpha, beta and a
column-major C.  The seed is fixed, so a failure reproduces.
"""
import numpy as np
import pytest
import torch

from dense_tiled_gemm_04_gb300 import native
from dense_tiled_gemm_04_gb300.workloads import make_inputs, round_up

import oracle
from test_gpu_epilogue import guard_ok, int_codes, run_ex
from test_gpu_parity import assert_exact, assert_guard, gpu_gemm

pytestmark = pytest.mark.gpu

CONFIGS = [native.CONFIG_AUTO, native.CONFIG_128x256, native.CONFIG_128x128, native.CONFIG_128x64,
           native.CONFIG_256x256]


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


def draw_case(rng):
    dim = lambda hi: int(np.exp(rng.uniform(0.0, np.log(hi))))  # noqa: E731  log-uniform in [1, hi)
    return dict(M=dim(1100), N=dim(1100), K=dim(700), layout=str(rng.choice(["NN", "TN"])),
                dtype=str(rng.choice(["f16", "bf16"])), config=int(rng.choice(CONFIGS)),
                stream_k=int(rng.integers(0, 2)), group=int(rng.choice([1, 2, 8, 64])),
                max_ctas=int(rng.choice([0, 0, 7, 40])), k_snake=int(rng.integers(0, 2)))


def with_options(g, case, fn):
    g.set_option(native.OPT_CONFIG, case["config"])
    g.set_option(native.OPT_STREAM_K, case["stream_k"])
    g.set_option(native.OPT_RASTER_GROUP, case["group"])
    g.set_option(native.OPT_MAX_CTAS, case["max_ctas"])
    g.set_option(native.OPT_K_SNAKE, case["k_snake"])
    try:
        return fn()
    finally:
        g.set_option(native.OPT_CONFIG, native.CONFIG_AUTO)
        g.set_option(native.OPT_STREAM_K, 1)
        g.set_option(native.OPT_RASTER_GROUP, 0)
        g.set_option(native.OPT_MAX_CTAS, 0)
        g.set_option(native.OPT_K_SNAKE, 1)


@pytest.mark.parametrize("chunk", range(4))
def test_random_shapes_and_launch_options(g, chunk):
    rng = np.random.default_rng(1000 + chunk)
    for i in range(12):
        c = draw_case(rng)
        M, N, K, layout, dtype = c["M"], c["N"], c["K"], c["layout"], c["dtype"]
        A, B = make_inputs(M, N, K, layout, dtype, "int", seed=2000 + 12 * chunk + i)
        got, buf = with_options(g, c, lambda: gpu_gemm(g, A, B, layout, dtype, extra_rows=3, ldc_pad=8))
        assert_guard(buf, M, N)
        assert_exact(got, oracle.gemm(A, B, layout, dtype), f"case {c}")


@pytest.mark.parametrize("chunk", range(2))
def test_random_epilogues(g, chunk):
    rng = np.random.default_rng(3000 + chunk)
    for i in range(12):
        c = draw_case(rng)
        M, N, K, layout, dtype = c["M"], c["N"], c["K"], c["layout"], c["dtype"]
        alpha = float(rng.choice([1.0, 2.0, -1.0]))
        beta = float(rng.choice([0.0, 1.0, -2.0]))
        col_major = int(rng.integers(0, 2))
        bcols = N if layout == "NN" else K
        A, B = make_inputs(M, N, K, layout, dtype, "int", seed=4000 + 12 * chunk + i, lda=round_up(K, 8),
                           ldb=round_up(bcols, 8))
        C0 = int_codes(M, N, dtype, 5000 + 12 * chunk + i)
        got, out, (r, cc) = with_options(g, c, lambda: run_ex(g, A, B, layout, dtype, alpha, beta, col_major, C0))
        assert guard_ok(out, r, cc), f"write outside the C window: case {c}"
        want = oracle.gemm_axpby(A, B, layout, dtype, alpha, beta, C0)
        assert_exact(got, want, f"case {c} alpha={alpha} beta={beta} col_major={col_major}")


def draw_8bit_case(rng):
    c = draw_case(rng)
    c.update(in_dtype=str(rng.choice(["e4m3", "e5m2"])), out=str(rng.choice(["f16", "bf16"])),
             alpha=float(rng.choice([1.0, 0.5, 2.0])), beta=float(rng.choice([0.0, 1.0])),
             col_major=int(rng.integers(0, 2)))
    return c


def test_random_8bit_operands_with_tensor_and_block_scales(g):
    from test_gpu_fp8 import factor, int_c, run8
    from test_gpu_mx import run_mx, scales

    rng = np.random.default_rng(6000)
    for i in range(16):
        c = draw_8bit_case(rng)
        M, N, K, layout = c["M"], c["N"], c["K"], c["layout"]
        A, B = make_inputs(M, N, K, layout, c["in_dtype"], "int", seed=6100 + i)
        C0 = int_c(M, N, c["out"], 6200 + i)
        kw = dict(alpha=c["alpha"], beta=c["beta"], col_major=bool(c["col_major"]), c_init=C0)
        if i % 2 == 0:  # per-tensor scales, gemm_run_ex
            got, guard = with_options(g, c, lambda: run8(g, A, B, layout, c["out"], scale_a=0.5, scale_b=2.0, **kw))
            want = oracle.gemm_typed(A, B, layout, c["in_dtype"], c["out"], alpha=factor(c["alpha"], 0.5, 2.0),
                                     beta=c["beta"], Cin=C0)
        else:  # E8M0 block scales, gemm_run_mx
            sa, sb = scales(M, K, 2, seed=6300 + i), scales(N, K, 2, seed=6400 + i)
            got, guard = with_options(g, c, lambda: run_mx(g, A, B, sa, sb, layout, c["out"], **kw))
            want = oracle.gemm_blockscaled(A, B, sa, sb, layout, c["in_dtype"], c["out"], alpha=c["alpha"],
                                           beta=c["beta"], Cin=C0)
        assert guard, f"write outside the C window: case {c}"
        assert_exact(got, want, f"case {i} {c}")


def test_random_sparse_operands(g):
    from dense_tiled_gemm_04_gb300.workloads import prune_24
    from test_gpu_sparse import compress, run_sp

    rng = np.random.default_rng(7000)
    for i in range(12):
        c = draw_case(rng)
        M, N, layout, dtype = c["M"], c["N"], c["layout"], c["dtype"]
        K = 4 * max(1, c["K"] // 4)  # a 2:4 A needs K in groups of four
        alpha, beta = float(rng.choice([1.0, 2.0])), float(rng.choice([0.0, -1.0]))
        col_major = int(rng.integers(0, 2))
        A, B = make_inputs(M, N, K, layout, dtype, "int", seed=7100 + i)
        A = prune_24(A, seed=7200 + i)
        C0 = int_codes(M, N, dtype, 7300 + i)
        Ac, meta, bad = compress(g, A)
        assert bad == 0
        got, guard = with_options(g, c, lambda: run_sp(g, Ac, meta, B, layout, dtype, alpha=alpha, beta=beta,
                                                       col_major=bool(col_major), c_init=C0))
        assert guard, f"write outside the C window: case {c}"
        assert_exact(got, oracle.gemm_axpby(A, B, layout, dtype, alpha, beta, C0), f"case {i} {c}")

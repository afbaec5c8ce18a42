"""Pins for the CPU oracle, against what the pages and the mathematics fix.

No GPU.  Each test checks the oracle against something other than itself: values the
pages print (``tests/golden``), closed forms, exhaustive comparison with library casts,
identity/permutation matrices, and an independent numpy fp64 matmul on small shapes.
"""
import itertools

import numpy as np
import pytest
import torch

from conftest import read_golden, read_shape_cases
from dense_tiled_gemm_04_gb300.workloads import make_inputs

import oracle
from oracle import tiled


def _f64(x):
    """fp64 values of a 16-bit torch tensor (torch's widening cast; exact)."""
    return x.to(torch.float64).numpy()


# ------------------------------------------------------------------ codecs


@pytest.mark.parametrize("dtype,tdt", [("f16", torch.float16), ("bf16", torch.bfloat16)])
def test_decode_every_code_matches_torch(dtype, tdt):
    codes = np.arange(65536, dtype=np.uint16)
    mine = oracle.decode(codes, dtype)
    ref = torch.from_numpy(codes.view(np.int16)).view(tdt).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(mine[~nan]), np.signbit(ref[~nan]))


def _sweep_values(dtype: str, tdt) -> np.ndarray:
    """fp32-representable test points: every finite code, every midpoint between
    neighbours (ties), midpoints +-1 fp32 ulp, random log-uniform values, overflow edges."""
    codes = np.arange(65536, dtype=np.uint16)
    vals = torch.from_numpy(codes.view(np.int16)).view(tdt).to(torch.float64).numpy()
    fin = np.sort(np.unique(vals[np.isfinite(vals)]))
    mids = (fin[:-1] + fin[1:]) / 2  # exact in fp64 and in fp32 (one extra bit)
    mids32 = mids.astype(np.float32)
    assert np.array_equal(mids32.astype(np.float64), mids)
    up = np.nextafter(mids32, np.float32(np.inf)).astype(np.float64)
    dn = np.nextafter(mids32, np.float32(-np.inf)).astype(np.float64)
    rng = np.random.default_rng(123)
    rnd = (rng.choice([-1.0, 1.0], 400_000) * np.exp2(rng.uniform(-140, 127.9, 400_000))).astype(np.float32)
    big = np.array([6.5504e4, 6.5519e4, 6.552e4, 6.5536e4, 1e5, 3.3895e38, 3.39e38, 3.4e38], dtype=np.float32)
    allv = np.concatenate([fin, mids, up, dn, rnd.astype(np.float64), big.astype(np.float64),
                           -big.astype(np.float64), [0.0, -0.0]])
    return allv.astype(np.float32).astype(np.float64)  # all exactly fp32


@pytest.mark.parametrize("dtype,tdt", [("f16", torch.float16), ("bf16", torch.bfloat16)])
def test_encode_matches_torch_rne_cast(dtype, tdt):
    # torch's fp32 -> fp16/bf16 cast rounds to nearest even with overflow to inf: a
    # library routine the oracle's own encoder must agree with on every fp32 input.
    x = _sweep_values(dtype, tdt)
    mine = oracle.encode(x, dtype)
    ref = torch.from_numpy(x.astype(np.float32)).to(tdt).view(torch.int16).numpy().view(np.uint16)
    bad = np.nonzero(mine != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches, e.g. x={x[bad[:5]]} mine={mine[bad[:5]]} torch={ref[bad[:5]]}"


def test_encode_ties_to_even_closed_form():
    # 2049 lies halfway between the fp16 neighbours 2048 and 2050: ties go to the even code.
    assert oracle.decode(oracle.encode([2049.0, 2051.0, 2050.0], "f16"), "f16").tolist() == [2048.0, 2052.0, 2050.0]
    # fp16 max is 65504; 65520 is the halfway point to 65536, which overflows.
    assert np.isinf(oracle.decode(oracle.encode([65520.0], "f16"), "f16"))[0]
    assert oracle.decode(oracle.encode([65519.0], "f16"), "f16")[0] == 65504.0
    # bf16 keeps 8 significant bits: 257 is a tie between 256 and 258 -> 256.
    assert oracle.decode(oracle.encode([257.0, 259.0], "bf16"), "bf16").tolist() == [256.0, 260.0]


# ------------------------------------------------------------------ the pages' worked example


def _shape_str_levels(levels):
    return [tuple(l) for l in levels]


def test_arrangement_shapes_match_page():
    cases = read_shape_cases("arrangement_shapes.txt")
    assert cases, "fixture empty"
    for (M, N, K, BM, BN, BK), expected in cases.items():
        got = tiled.arrangement_shapes(M, N, K, BM, BN, BK)
        for label, levels in expected.items():
            assert _shape_str_levels(got[label]) == levels, (label, got[label], levels)


def test_worked_example_grid_and_block_identities():
    g = read_golden("worked_example.txt")
    M, N, K, BM, BN, BK = g["M"], g["N"], g["K"], g["BM"], g["BN"], g["BK"]
    TM, TN, KB = tiled.grid(M, N, K, BM, BN, BK)
    assert (TM, TN) == g["grid"] and KB == g["k_blocks"] and TM * TN == g["programs"]

    A, B = make_inputs(M, N, K, "NN", "f16", "int", seed=0)
    A64, B64 = _f64(A), _f64(B)
    i, j = g["program"]
    p = g["p"]
    # lhs[p][r,t] = A[i*BM+r, p*BK+t] and rhs[p][t,s] = B[p*BK+t, j*BN+s]
    r0, r1 = g["a_rows"]
    c0, c1 = g["a_cols"]
    assert np.array_equal(tiled.lhs_block(A64, i, p, BM, BK), A64[r0:r1, c0:c1])
    r0, r1 = g["b_rows"]
    c0, c1 = g["b_cols"]
    assert np.array_equal(tiled.rhs_block(B64, j, p, BK, BN), B64[r0:r1, c0:c1])

    # The oracle's direct sum equals the tile-by-tile K-block sum exactly (integers).
    codes, direct = oracle.gemm(A, B, "NN", "f16", want_f64=True)
    blocked = tiled.tiled_gemm(A64, B64, BM, BN, BK)
    assert np.array_equal(direct, blocked)
    # C_tile[1,2] = sum_p A[i*BM:, p*BK:] B[p*BK:, j*BN:] covers C[64:128, 128:192]
    cr0, cr1 = g["c_rows"]
    cc0, cc1 = g["c_cols"]
    tile = sum(A64[cr0:cr1, q * BK:(q + 1) * BK] @ B64[q * BK:(q + 1) * BK, cc0:cc1] for q in range(KB))
    assert np.array_equal(direct[cr0:cr1, cc0:cc1], tile)
    # BK = 32 (§8 exercise one): 6 K blocks, same result
    assert tiled.grid(M, N, K, 64, 64, 32)[2] == 6
    assert np.array_equal(direct, tiled.tiled_gemm(A64, B64, 64, 64, 32))


def test_worked_example_random_inputs_blocked_vs_direct():
    # Uniform inputs (the worked example's own distribution): fp64 sums of fp16
    # products are exact here, so blocking must not change a single bit.
    A, B = make_inputs(128, 256, 192, "NN", "f16", "uniform", seed=0)
    codes, direct = oracle.gemm(A, B, "NN", "f16", want_f64=True)
    blocked = tiled.tiled_gemm(_f64(A), _f64(B), 64, 64, 64)
    np.testing.assert_allclose(direct, blocked, rtol=0, atol=1e-12)
    assert np.array_equal(codes, oracle.encode(direct, "f16"))


@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_tail_all_ones_is_130(layout):
    g = read_golden("tail_allones.txt")
    M, N, K, BM, BN, BK = g["M"], g["N"], g["K"], g["BM"], g["BN"], g["BK"]
    TM, TN, KB = tiled.grid(M, N, K, BM, BN, BK)
    assert (TM, TN) == g["grid"] and KB == g["k_blocks"]
    rows, cols, kv = tiled.tail_valid_counts(M, N, K, BM, BN, BK)
    assert (rows, cols) == g["corner_valid"] and kv == g["last_k_valid"]

    A, B = make_inputs(M, N, K, layout, "f16", "ones", seed=0)
    C = oracle.decode(oracle.gemm(A, B, layout, "f16"), "f16")
    assert C.shape == (M, N) and np.all(C == g["allones_value"])
    # The mistake the page's exercise is built to catch: a K loop one block short.
    Bl = _f64(B) if layout == "NN" else _f64(B).T
    short = tiled.tiled_gemm(_f64(A), Bl, BM, BN, BK, drop_last_k_block=True)
    assert np.all(short == g["allones_value_without_last_k_tile"])
    assert np.all(tiled.tiled_gemm(_f64(A), Bl, BM, BN, BK) == g["allones_value"])


def test_fp32_accumulation_example():
    g = read_golden("fp32_accumulation.txt")
    a = np.array([g["a_row"]], dtype=np.float32)
    b = np.array([g["b_col"]], dtype=np.float32).T
    A = torch.from_numpy(a).to(torch.float16)
    B = torch.from_numpy(b).to(torch.float16)
    C = oracle.decode(oracle.gemm(A, B, "NN", "f16"), "f16")
    assert C[0, 0] == g["fp16_output"] == g["fp32_accumulate"]
    # The same sum rounded back to fp16 after every add stays at 2048.
    acc = 0.0
    for x, y in zip(g["a_row"], g["b_col"]):
        acc = float(oracle.decode(oracle.encode([acc + x * y], "f16"), "f16")[0])
    assert acc == g["fp16_accumulate"]


# ------------------------------------------------------------------ closed forms


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_identity_and_permutation(layout, dtype):
    M, K = 37, 29
    A, _ = make_inputs(M, K, K, layout, dtype, "uniform", seed=5)
    tdt = A.dtype
    eye = torch.eye(K, dtype=tdt)
    assert np.array_equal(oracle.gemm(A, eye, layout, dtype), oracle._codes(A))
    perm = torch.randperm(K, generator=torch.Generator().manual_seed(9))
    P = torch.zeros(K, K, dtype=tdt)
    P[perm, torch.arange(K)] = 1  # Beff = P: (A P)[:, j] = A[:, perm[j]]
    Bstored = P if layout == "NN" else P.T.contiguous()
    got = oracle.gemm(A, Bstored, layout, dtype)
    assert np.array_equal(got, oracle._codes(A)[:, perm.numpy()])


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_tn_equals_nn_of_transposed_b(dtype):
    A, B = make_inputs(23, 41, 19, "NN", dtype, "normal", seed=11)
    nn = oracle.gemm(A, B, "NN", dtype)
    tn = oracle.gemm(A, B.T.contiguous(), "TN", dtype)
    assert np.array_equal(nn, tn)


SIZES = [1, 2, 3, 5, 8, 9, 15, 16, 17, 63, 64, 65, 127, 128, 129]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_brute_force_against_numpy_f64(dtype):
    """Independent numpy fp64 matmul on every (M, N, K) from a size set: equal sums
    (within fp64 reordering) and, on integer data, identical rounded codes."""
    rng = np.random.default_rng(7)
    combos = list(itertools.product(SIZES, repeat=3))
    rng.shuffle(combos)
    for idx, (M, N, K) in enumerate(combos[:400]):
        layout = "NN" if idx % 2 == 0 else "TN"
        dist = "int" if idx % 3 == 0 else "normal"
        A, B = make_inputs(M, N, K, layout, dtype, dist, seed=idx)
        codes, f64 = oracle.gemm(A, B, layout, dtype, want_f64=True)
        Bl = _f64(B) if layout == "NN" else _f64(B).T
        ref = _f64(A) @ Bl
        np.testing.assert_allclose(f64, ref, rtol=1e-13, atol=1e-13, err_msg=str((M, N, K, layout)))
        if dist == "int":
            assert np.array_equal(f64, ref)
            assert np.array_equal(codes, oracle.encode(ref, dtype))
            if dtype == "f16":  # numpy's own fp64 -> fp16 cast, a separate rounding routine
                assert np.array_equal(codes, ref.astype(np.float16).view(np.uint16))


def test_blocked_equals_direct_on_small_tiles():
    """Tile-by-tile formulation with small tiles vs the direct sum, ragged in M, N, K."""
    for (M, N, K) in [(1, 1, 1), (5, 9, 3), (9, 8, 17), (16, 15, 16), (17, 17, 9)]:
        A, B = make_inputs(M, N, K, "NN", "f16", "int", seed=M * 100 + N + K)
        direct = oracle.gemm(A, B, "NN", "f16", want_f64=True)[1]
        for (BM, BN, BK) in [(4, 8, 4), (8, 4, 16), (16, 16, 8)]:
            assert np.array_equal(direct, tiled.tiled_gemm(_f64(A), _f64(B), BM, BN, BK))


@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_padded_leading_dimensions(layout):
    M, N, K = 19, 21, 13
    A, B = make_inputs(M, N, K, layout, "f16", "normal", seed=3)
    Ap, Bp = make_inputs(M, N, K, layout, "f16", "normal", seed=3, lda=24, ldb=32)
    assert torch.isnan(Ap.as_strided((M, 24), (24, 1))[:, K:]).all()  # NaN padding really there
    assert np.array_equal(oracle.gemm(A, B, layout, "f16"), oracle.gemm(Ap, Bp, layout, "f16"))


@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_elems_and_rows_agree_with_full(layout):
    M, N, K = 70, 90, 50
    A, B = make_inputs(M, N, K, layout, "bf16", "uniform", seed=21)
    full = oracle.gemm(A, B, layout, "bf16")
    rng = np.random.default_rng(0)
    ms, ns = rng.integers(0, M, 200), rng.integers(0, N, 200)
    assert np.array_equal(oracle.gemm_elems(A, B, layout, "bf16", ms, ns), full[ms, ns])
    rows = np.array([0, 69, 33])
    assert np.array_equal(oracle.gemm_rows(A, B, layout, "bf16", rows)[0], full[rows])


def test_k_zero_is_the_empty_sum():
    A = torch.zeros(4, 0, dtype=torch.float16)
    B = torch.zeros(0, 6, dtype=torch.float16)
    C = oracle.gemm(A, B, "NN", "f16")
    assert C.shape == (4, 6) and np.all(C == 0)


def test_overflow_rounds_to_inf():
    A = torch.full((1, 4), 200.0, dtype=torch.float16)
    B = torch.full((4, 1), 200.0, dtype=torch.float16)  # 4 * 40000 = 160000 > 65504
    C = oracle.decode(oracle.gemm(A, B, "NN", "f16"), "f16")
    assert np.isposinf(C[0, 0])


# ------------------------------------------------------------------ alpha / beta (C = alpha A·B + beta C)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_axpby_closed_forms(layout, dtype):
    M, N, K = 33, 47, 29
    A, B = make_inputs(M, N, K, layout, dtype, "int", seed=31)
    Cin, _ = make_inputs(M, N, N, "NN", dtype, "normal", seed=32)  # any M x N codes
    plain = oracle.gemm(A, B, layout, dtype)
    # alpha = 1, beta = 0 is the plain product (Cin not read: pass garbage-free None)
    assert np.array_equal(oracle.gemm_axpby(A, B, layout, dtype, 1.0, 0.0), plain)
    # alpha = 0, beta = 1 returns Cin unchanged (every code re-rounds to itself)
    assert np.array_equal(oracle.gemm_axpby(A, B, layout, dtype, 0.0, 1.0, Cin), oracle._codes(Cin))
    # alpha = 2 doubles the exact sum (a power-of-two scale is exact before the rounding)
    codes, f64 = oracle.gemm_axpby(A, B, layout, dtype, 2.0, 0.0, want_f64=True)
    _, base = oracle.gemm(A, B, layout, dtype, want_f64=True)
    assert np.array_equal(f64, 2.0 * base) and np.array_equal(codes, oracle.encode(2.0 * base, dtype))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_axpby_accumulate_form_against_numpy(dtype):
    """C += A·B (alpha = beta = 1) twice, against an independent numpy fp64 evaluation;
    small integers keep every value exact, so the codes must match bit for bit."""
    M, N, K = 40, 24, 12
    A, B = make_inputs(M, N, K, "TN", dtype, "int", seed=33)
    C0, _ = make_inputs(M, N, N, "NN", dtype, "int", seed=34)
    A64, B64 = A.to(torch.float64).numpy(), B.to(torch.float64).numpy().T
    C1 = oracle.gemm_axpby(A, B, "TN", dtype, 1.0, 1.0, C0)
    C2 = oracle.gemm_axpby(A, B, "TN", dtype, 1.0, 1.0, C1)
    ref2 = 2.0 * (A64 @ B64) + C0.to(torch.float64).numpy()
    assert np.array_equal(oracle.decode(C2, dtype), ref2)
    # beta = -1 with Cin = A·B cancels exactly
    AB = oracle.gemm(A, B, "TN", dtype)
    assert np.all(oracle.decode(oracle.gemm_axpby(A, B, "TN", dtype, 1.0, -1.0, AB), dtype) == 0.0)


def test_axpby_general_scalars_match_numpy_within_rounding():
    M, N, K = 20, 30, 50
    A, B = make_inputs(M, N, K, "NN", "f16", "normal", seed=35)
    Cin, _ = make_inputs(M, N, N, "NN", "f16", "normal", seed=36)
    _, f64 = oracle.gemm_axpby(A, B, "NN", "f16", 0.75, -1.25, Cin, want_f64=True)
    ref = 0.75 * (A.to(torch.float64).numpy() @ B.to(torch.float64).numpy()) - 1.25 * Cin.to(torch.float64).numpy()
    np.testing.assert_allclose(f64, ref, rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------ 8-bit inputs


@pytest.mark.parametrize("fmt,tdt", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_fp8_decode_every_code_matches_torch(fmt, tdt):
    codes = np.arange(256, dtype=np.uint16)
    mine = oracle.decode(codes, fmt)
    ref = torch.from_numpy(codes.astype(np.uint8)).view(tdt).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.array_equal(np.signbit(mine[~nan]), np.signbit(ref[~nan]))


def test_fp8_closed_forms():
    # E4M3 largest finite 448 (0x7e), smallest subnormal 2^-9 (0x01), NaN 0x7f; E5M2 inf 0x7c.
    assert oracle.decode([0x7E, 0x01, 0x38], "e4m3").tolist() == [448.0, 2.0 ** -9, 1.0]
    assert np.isnan(oracle.decode([0x7F], "e4m3")[0])
    assert oracle.decode([0x7B, 0x01, 0x3C], "e5m2").tolist() == [57344.0, 2.0 ** -16, 1.0]
    assert np.isposinf(oracle.decode([0x7C], "e5m2")[0])


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("out", ["f16", "bf16"])
@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_fp8_gemm_equals_16bit_gemm_on_exact_values(fmt, out, layout):
    # Integers in {-2..2} are exact in every format: the 8-bit product must equal the
    # 16-bit product of the same values, code for code.
    M, N, K = 37, 45, 70
    A8, B8 = make_inputs(M, N, K, layout, fmt, "int", seed=41)
    A16, B16 = A8.to(torch.float32).to(torch.bfloat16 if out == "bf16" else torch.float16), \
        B8.to(torch.float32).to(torch.bfloat16 if out == "bf16" else torch.float16)
    assert np.array_equal(oracle.gemm_typed(A8, B8, layout, fmt, out), oracle.gemm(A16, B16, layout, out))


def test_fp8_scales_and_random_values():
    M, N, K = 30, 40, 64
    A, B = make_inputs(M, N, K, "TN", "e4m3", "normal", seed=42)
    sa, sb = 0.5, 8.0  # powers of two: the scaled sum is exact before the rounding
    codes, f64 = oracle.gemm_typed(A, B, "TN", "e4m3", "bf16", alpha=sa * sb, want_f64=True)
    ref = A.to(torch.float64).numpy() @ B.to(torch.float64).numpy().T
    np.testing.assert_allclose(f64, sa * sb * ref, rtol=1e-13, atol=1e-13)
    assert np.array_equal(codes, oracle.encode(f64, "bf16"))
    # beta folds in a 16-bit C of the output type
    Cin, _ = make_inputs(M, N, N, "NN", "bf16", "int", seed=43)
    _, f64b = oracle.gemm_typed(A, B, "TN", "e4m3", "bf16", alpha=1.0, beta=-1.0, Cin=Cin, want_f64=True)
    np.testing.assert_allclose(f64b, ref - Cin.to(torch.float64).numpy(), rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------ 8-bit inputs, per-tile scales


def test_e8m0_scale_codes():
    # E8M0 (the OCP microscaling scale format): 2^(e - 127), e = 255 is NaN.
    assert oracle.e8m0(127) == 1.0 and oracle.e8m0(128) == 2.0 and oracle.e8m0(126) == 0.5
    assert oracle.e8m0(0) == 2.0 ** -127 and oracle.e8m0(254) == 2.0 ** 127
    assert np.isnan(oracle.e8m0(255))
    if hasattr(torch, "float8_e8m0fnu"):
        codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
        ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
        mine = np.array([oracle.e8m0(e) for e in range(256)])
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(mine), nan)
        assert np.array_equal(mine[~nan], ref[~nan])


def _expand(s: np.ndarray, K: int) -> np.ndarray:
    """Per-element scale 2^(s[:, k // 32] - 127): the scales written out element by element."""
    e = np.repeat(s.astype(np.int64), 32, axis=1)[:, :K]
    return np.ldexp(1.0, e - 127)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_blockscaled_unit_scales_equal_the_unscaled_contraction(fmt, layout):
    M, N, K = 19, 23, 70  # three K blocks, the last one 6 long
    A, B = make_inputs(M, N, K, layout, fmt, "normal", seed=51)
    nb = -(-K // 32)
    one_a, one_b = np.full((M, nb), 127, np.uint8), np.full((N, nb), 127, np.uint8)
    for out in ("f16", "bf16"):
        got = oracle.gemm_blockscaled(A, B, one_a, one_b, layout, fmt, out)
        assert np.array_equal(got, oracle.gemm_typed(A, B, layout, fmt, out))


@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_blockscaled_row_and_column_scales_closed_form(layout):
    # Scales constant along K factor out of the sum: C = 2^r_m * 2^c_n * (A·B)[m, n].
    M, N, K = 21, 17, 96
    A, B = make_inputs(M, N, K, layout, "e4m3", "int", seed=52)
    rng = np.random.default_rng(53)
    r, c = rng.integers(-3, 4, M), rng.integers(-3, 4, N)
    sa = np.repeat((127 + r)[:, None], 3, axis=1).astype(np.uint8)
    sb = np.repeat((127 + c)[:, None], 3, axis=1).astype(np.uint8)
    _, f64 = oracle.gemm_blockscaled(A, B, sa, sb, layout, "e4m3", "bf16", want_f64=True)
    a, b = A.to(torch.float64).numpy(), B.to(torch.float64).numpy()
    ab = a @ (b if layout == "NN" else b.T)
    assert np.array_equal(f64, np.ldexp(1.0, r)[:, None] * np.ldexp(1.0, c)[None, :] * ab)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_blockscaled_against_dequantise_then_multiply(fmt, layout):
    # The tile-by-tile form (contract a 32-long K block, scale, accumulate) against the other
    # way round: scale every element of A and B, then one numpy fp64 product.  M != N and a
    # ragged last block, so an index of the wrong operand, the wrong block or a dropped tail
    # block all show.
    M, N, K = 27, 41, 150
    A, B = make_inputs(M, N, K, layout, fmt, "normal", seed=54)
    nb = -(-K // 32)
    rng = np.random.default_rng(55)
    sa = rng.integers(120, 135, (M, nb)).astype(np.uint8)
    sb = rng.integers(120, 135, (N, nb)).astype(np.uint8)
    _, f64 = oracle.gemm_blockscaled(A, B, sa, sb, layout, fmt, "f16", want_f64=True)
    a = A.to(torch.float64).numpy() * _expand(sa, K)
    bt = (B.to(torch.float64).numpy() if layout == "TN" else B.to(torch.float64).numpy().T) * _expand(sb, K)
    ref = a @ bt.T
    np.testing.assert_allclose(f64, ref, rtol=1e-12, atol=1e-30)


def test_blockscaled_one_block_scale_changes_one_partial():
    # Raising one A scale by one step doubles exactly that block's share of the row.
    M, N, K = 6, 9, 96
    A, B = make_inputs(M, N, K, "TN", "e4m3", "int", seed=56)
    sa, sb = np.full((M, 3), 127, np.uint8), np.full((N, 3), 127, np.uint8)
    _, base = oracle.gemm_blockscaled(A, B, sa, sb, "TN", "e4m3", "bf16", want_f64=True)
    sa2 = sa.copy()
    sa2[4, 1] = 128
    _, f64 = oracle.gemm_blockscaled(A, B, sa2, sb, "TN", "e4m3", "bf16", want_f64=True)
    a, b = A.to(torch.float64).numpy(), B.to(torch.float64).numpy()
    block1 = a[4, 32:64] @ b[:, 32:64].T
    expect = base.copy()
    expect[4] += block1
    assert np.array_equal(f64, expect)


def test_blockscaled_nan_scale_and_epilogue():
    M, N, K = 8, 12, 64
    A, B = make_inputs(M, N, K, "NN", "e5m2", "int", seed=57)
    sa, sb = np.full((M, 2), 127, np.uint8), np.full((N, 2), 127, np.uint8)
    sa[3, 1] = 255
    got = oracle.decode(oracle.gemm_blockscaled(A, B, sa, sb, "NN", "e5m2", "f16"), "f16")
    assert np.all(np.isnan(got[3])) and not np.isnan(np.delete(got, 3, axis=0)).any()
    sa[3, 1] = 127
    Cin, _ = make_inputs(M, N, N, "NN", "f16", "int", seed=58)
    _, f64 = oracle.gemm_blockscaled(A, B, sa, sb, "NN", "e5m2", "f16", alpha=0.5, beta=-1.0, Cin=Cin,
                                     want_f64=True)
    ref = 0.5 * (A.to(torch.float64).numpy() @ B.to(torch.float64).numpy()) - Cin.to(torch.float64).numpy()
    assert np.array_equal(f64, ref)


# ------------------------------------------------------------------ 2:4 structured sparsity
from dense_tiled_gemm_04_gb300.workloads import prune_24  # noqa: E402


def _f16_codes(vals):
    return torch.tensor(vals, dtype=torch.float16).view(torch.int16).numpy().view(np.uint16)


def test_sparse24_compress_closed_forms():
    # Groups: [0,5,0,7] -> (1,3); all zero -> (0,1); [3,0,0,0] -> (0,1); [0,0,0,9] -> (0,3);
    # [-0,0,6,0] -> (0,2) (negative zero is zero); [1,2,3,4] -> (0,1), counted as a violation;
    # [0,8,2,0] -> (1,2); [0,0,4,4] -> (2,3).
    row = [0, 5, 0, 7, 0, 0, 0, 0, 3, 0, 0, 0, 0, 0, 0, 9, -0.0, 0, 6, 0, 1, 2, 3, 4, 0, 8, 2, 0, 0, 0, 4, 4,
           0, 0, 1, 0]
    A = _f16_codes([row])
    Ac, E, bad = oracle.sparse24_compress(A)
    assert bad == 1
    assert oracle.decode(Ac, "f16").tolist() == [[5, 7, 0, 0, 3, 0, 0, 9, -0.0, 6, 1, 2, 8, 2, 4, 4, 0, 1]]
    pairs = [(1, 3), (0, 1), (0, 1), (0, 3), (0, 2), (0, 1), (1, 2), (2, 3), (0, 2)]
    nibbles = [a | (b << 2) for a, b in pairs]
    words = [sum(n << (4 * i) for i, n in enumerate(nibbles[:8])), nibbles[8]]
    assert E.tolist() == [words]
    assert E.dtype == np.uint32 and words[0] == 0xE948C44D  # nibbles D,4,4,C,8,4,9,E from the low end


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("layout", ["NN", "TN"])
def test_sparse24_contraction_equals_dense_product(layout, dtype):
    # The sparse form (kept values times the B rows the metadata names) against the plain
    # dense product of the 2:4 matrix: integer data is exact in fp64 whatever the order.
    M, N, K = 33, 47, 100  # 25 groups: the last metadata word holds one group
    A, B = make_inputs(M, N, K, layout, dtype, "int", seed=91)
    A = prune_24(A, seed=92)
    Ac, E, bad = oracle.sparse24_compress(A)
    assert bad == 0 and Ac.shape == (M, K // 2) and E.shape == (M, 4)
    codes, f64 = oracle.gemm_sparse24(Ac, E, B, layout, dtype, want_f64=True)
    dense = oracle.gemm_rows(A, B, layout, dtype, np.arange(M), want_f64=True)
    assert np.array_equal(codes, dense[0])
    assert np.array_equal(f64, dense[1])
    a, b = A.to(torch.float64).numpy(), B.to(torch.float64).numpy()
    assert np.array_equal(f64, a @ (b if layout == "NN" else b.T))


def test_sparse24_normal_values_and_epilogue():
    M, N, K = 40, 24, 64
    A, B = make_inputs(M, N, K, "TN", "bf16", "normal", seed=93)
    A = prune_24(A, seed=94)
    Ac, E, _ = oracle.sparse24_compress(A)
    Cin, _ = make_inputs(M, N, N, "NN", "bf16", "int", seed=95)
    _, f64 = oracle.gemm_sparse24(Ac, E, B, "TN", "bf16", alpha=0.5, beta=-2.0, Cin=Cin, want_f64=True)
    ref = 0.5 * (A.to(torch.float64).numpy() @ B.to(torch.float64).numpy().T) - 2.0 * Cin.to(torch.float64).numpy()
    np.testing.assert_allclose(f64, ref, rtol=1e-13, atol=1e-13)


def test_sparse24_metadata_selects_the_b_row():
    # One kept 1.0 at K position 4g + i of row m: row m of C is row 4g + i of B (NN).
    M, N, K = 4, 16, 64
    _, B = make_inputs(M, N, K, "NN", "f16", "int", seed=96)
    for m, k in [(0, 0), (1, 5), (2, 42), (3, 63)]:
        A = torch.zeros((M, K), dtype=torch.float16)
        A[m, k] = 1.0
        Ac, E, bad = oracle.sparse24_compress(A)
        assert bad == 0
        got = oracle.gemm_sparse24(Ac, E, B, "NN", "f16")
        assert np.array_equal(got[m], B[k].view(torch.int16).numpy().view(np.uint16))


def test_sparse24_violation_keeps_the_first_two():
    A = _f16_codes([[1, 2, 3, 0, 0, 0, 0, 0]])
    B = _f16_codes([[1], [10], [100], [1000], [0], [0], [0], [0]])
    Ac, E, bad = oracle.sparse24_compress(A)
    assert bad == 1
    assert oracle.decode(oracle.gemm_sparse24(Ac, E, B, "NN", "f16"), "f16").tolist() == [[21.0]]

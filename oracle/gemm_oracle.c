/*
 * CPU oracle for the tiled dense contraction C = A·B (fp16/bf16 in, wide accumulate,
 * fp16/bf16 out).  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg call it; the GPU library never does, and this file
 * shares no code, header, table or helper with it.
 *
 * What it computes (the plain definition, no blocking, no reordering):
 *
 *     C[m,n] = round_out( sum_{k<K} A[m,k] * Beff[k,n] )        (sum taken in fp64)
 *
 *   - "NineToothed GEMM 语法入门" (NineToothed GEMM syntax primer) §2 "from the
 *     symbolic layout to application": the accumulator starts at zero, every K block
 *     adds its product, and the output is assigned once.  §3 "tracing one read" gives
 *     the index identities lhs[p][r,t] = A[i*BM+r, p*BK+t], rhs[p][t,s] = B[p*BK+t, j*BN+s];
 *     summed over all p and t they reduce to the single sum over k written above.
 *   - same page §4: the result must contain the products over the whole K range.
 *   - same page §5 "how tail blocks take part": reads outside M/N/K contribute zero
 *     and writes outside M x N are suppressed, so only the real indices appear here.
 *   - same page §6 "what float32 accumulation keeps": inputs and outputs are 16-bit,
 *     the accumulator is wider and the value is rounded once when written back.  This
 *     oracle accumulates in fp64 (wider than the kernel's fp32) and rounds once,
 *     round-to-nearest-even, the IEEE default.
 *
 * Layouts (A is always M x K row-major with leading dimension lda):
 *   NN: B stored K x N row-major, Beff[k,n] = B[k*ldb + n]   (the page's B is (192, 256))
 *   TN: B stored N x K row-major, Beff[k,n] = B[n*ldb + k]   ("张量缩并：mma 语法", the
 *       one-warp kernel takes rhs as [N, K])
 *
 * Codecs are written from the IEEE 754 binary16 definition (1 sign, 5 exponent bits with
 * bias 15, 10 fraction bits) and from bfloat16 (1 sign, 8 exponent bits with bias 127,
 * 7 fraction bits).  Widening to fp64 is exact; narrowing rounds to nearest, ties to even,
 * overflows to +-inf and keeps subnormals.
 *
 * Compiled with -ffp-contract=off so that x86 and Arm builds perform the same roundings.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_LAYOUT_NN = 0, OR_LAYOUT_TN = 1 };
enum { OR_F16 = 0, OR_BF16 = 1, OR_E4M3 = 2, OR_E5M2 = 3 };

/* ---------------------------------------------------------------- decode */

double oracle_f16_to_f64(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1f;
    const int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);              /* subnormal: f * 2^(1-15-10) */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f | 0x400), e - 25); /* (1024+f) * 2^(e-15-10) */
    return sign ? -v : v;
}

double oracle_bf16_to_f64(uint16_t b)
{
    const int sign = (b >> 15) & 1;
    const int e = (b >> 7) & 0xff;
    const int f = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);             /* subnormal: f * 2^(1-127-7) */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f | 0x80), e - 134); /* (128+f) * 2^(e-127-7) */
    return sign ? -v : v;
}

/* 8-bit floats (inputs only), from their definitions:
 *   E4M3: 1 sign, 4 exponent bits (bias 7), 3 fraction bits; no infinities; exponent and
 *         fraction all ones (S.1111.111) is NaN; largest finite 448.
 *   E5M2: 1 sign, 5 exponent bits (bias 15), 2 fraction bits; IEEE-style inf and NaN. */
double oracle_e4m3_to_f64(uint8_t c)
{
    const int sign = (c >> 7) & 1;
    const int e = (c >> 3) & 0xf;
    const int f = c & 0x7;
    double v;
    if (e == 15 && f == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)f, -9);             /* subnormal: f * 2^(1-7-3) */
    else
        v = ldexp((double)(f | 0x8), e - 10); /* (8+f) * 2^(e-7-3) */
    return sign ? -v : v;
}

double oracle_e5m2_to_f64(uint8_t c)
{
    const int sign = (c >> 7) & 1;
    const int e = (c >> 2) & 0x1f;
    const int f = c & 0x3;
    double v;
    if (e == 0)
        v = ldexp((double)f, -16);            /* subnormal: f * 2^(1-15-2) */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f | 0x4), e - 17); /* (4+f) * 2^(e-15-2) */
    return sign ? -v : v;
}

/* ---------------------------------------------------------------- encode */

/* Round a non-negative integer-valued-or-not double n to the nearest integer,
 * ties to the even one.  n < 2^52 here, so floor and the difference are exact. */
static double round_half_even(double n)
{
    const double fl = floor(n);
    const double d = n - fl;
    if (d > 0.5) return fl + 1.0;
    if (d < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* Generic narrowing of x to a binary format with `mbits` fraction bits, minimum
 * normal exponent `emin`, largest finite value `maxv`.  Returns the rounded value
 * as a double (exactly representable in the target format) or +-inf. */
static double round_to_format(double x, int mbits, int emin, double maxv)
{
    const double a = fabs(x);
    if (a == 0.0 || isinf(a) || isnan(a)) return x;
    int e2;
    frexp(a, &e2);           /* a in [2^(e2-1), 2^e2) */
    int E = e2 - 1;          /* binade exponent of a */
    if (E < emin) E = emin;  /* subnormal binade shares the quantum of the smallest normal */
    const double q = ldexp(1.0, E - mbits);   /* spacing of representable values */
    const double r = round_half_even(a / q) * q;
    const double v = (r > maxv) ? INFINITY : r;
    return signbit(x) ? -v : v;
}

static uint16_t pack_format(double v, int mbits, int ebits, int emin)
{
    const uint16_t sign = signbit(v) ? (uint16_t)(1u << 15) : 0;
    const int bias = (1 << (ebits - 1)) - 1;
    const double a = fabs(v);
    if (isnan(v)) /* quiet NaN with the top fraction bit set */
        return (uint16_t)(((1u << ebits) - 1) << mbits | (1u << (mbits - 1)));
    if (isinf(a)) return (uint16_t)(sign | (((1u << ebits) - 1) << mbits));
    if (a == 0.0) return sign;
    if (a < ldexp(1.0, emin)) { /* subnormal: a = f * 2^(emin - mbits) */
        const double f = a / ldexp(1.0, emin - mbits);
        return (uint16_t)(sign | (uint16_t)f);
    }
    int e2;
    frexp(a, &e2);
    const int E = e2 - 1;
    const double frac = a / ldexp(1.0, E - mbits) - ldexp(1.0, mbits);
    return (uint16_t)(sign | (uint16_t)((E + bias) << mbits) | (uint16_t)frac);
}

uint16_t oracle_f64_to_f16(double x)
{
    return pack_format(round_to_format(x, 10, -14, 65504.0), 10, 5, -14);
}

uint16_t oracle_f64_to_bf16(double x)
{
    /* largest finite bfloat16: (2 - 2^-7) * 2^127 */
    return pack_format(round_to_format(x, 7, -126, ldexp(255.0, 120)), 7, 8, -126);
}

/* ---------------------------------------------------------------- GEMM */

/* Value of every input code; 8-bit formats use the low byte of the 16-bit code. */
static void build_table(double* t, int dtype)
{
    for (uint32_t c = 0; c < 65536u; ++c) {
        if (dtype == OR_E4M3)
            t[c] = oracle_e4m3_to_f64((uint8_t)(c & 0xffu));
        else if (dtype == OR_E5M2)
            t[c] = oracle_e5m2_to_f64((uint8_t)(c & 0xffu));
        else
            t[c] = (dtype == OR_BF16) ? oracle_bf16_to_f64((uint16_t)c) : oracle_f16_to_f64((uint16_t)c);
    }
}

/* One output row m of the fp64 accumulator: acc[n] for n < N. */
static void row_f64(const double* T, const uint16_t* A, const uint16_t* B, int64_t m,
                    int64_t N, int64_t K, int64_t lda, int64_t ldb, int layout, double* acc)
{
    const uint16_t* arow = A + m * lda;
    if (layout == OR_LAYOUT_NN) {
        for (int64_t n = 0; n < N; ++n) acc[n] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = T[arow[k]];
            const uint16_t* brow = B + k * ldb;
            for (int64_t n = 0; n < N; ++n) acc[n] += a * T[brow[n]];
        }
    } else {
        for (int64_t n = 0; n < N; ++n) {
            const uint16_t* bcol = B + n * ldb; /* column n of Beff is row n of the stored N x K array */
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) s += T[arow[k]] * T[bcol[k]];
            acc[n] = s;
        }
    }
}

/* Rows `rows[0..nrows)` of C.  If `out16` is non-null, writes the rounded 16-bit codes
 * (row i of the output at out16 + i*ldo); if `out64` is non-null, writes the unrounded
 * fp64 sums (row i at out64 + i*ldo).  Returns the number of threads used. */
int oracle_gemm_rows(const uint16_t* A, const uint16_t* B, int64_t N, int64_t K,
                     int64_t lda, int64_t ldb, int layout, int dtype,
                     const int64_t* rows, int64_t nrows,
                     uint16_t* out16, double* out64, int64_t ldo, int nthreads)
{
    double* T = (double*)malloc(65536 * sizeof(double));
    if (!T) return -1;
    build_table(T, dtype);
    int used = 1;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
    {
#pragma omp single
        used = omp_get_num_threads();
        double* acc = (double*)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nrows; ++i) {
            row_f64(T, A, B, rows[i], N, K, lda, ldb, layout, acc);
            for (int64_t n = 0; n < N; ++n) {
                if (out64) out64[i * ldo + n] = acc[n];
                if (out16) out16[i * ldo + n] = (dtype == OR_BF16) ? oracle_f64_to_bf16(acc[n])
                                                                    : oracle_f64_to_f16(acc[n]);
            }
        }
        free(acc);
    }
#else
    (void)nthreads;
    double* acc = (double*)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    for (int64_t i = 0; i < nrows; ++i) {
        row_f64(T, A, B, rows[i], N, K, lda, ldb, layout, acc);
        for (int64_t n = 0; n < N; ++n) {
            if (out64) out64[i * ldo + n] = acc[n];
            if (out16) out16[i * ldo + n] = (dtype == OR_BF16) ? oracle_f64_to_bf16(acc[n])
                                                                : oracle_f64_to_f16(acc[n]);
        }
    }
    free(acc);
#endif
    free(T);
    return used;
}

/* Individual elements (ms[i], ns[i]) of C, for sampled checks at sizes where whole rows
 * are too slow.  Same definition, one dot product per element. */
int oracle_gemm_elems(const uint16_t* A, const uint16_t* B, int64_t K, int64_t lda, int64_t ldb,
                      int layout, int dtype, const int64_t* ms, const int64_t* ns, int64_t count,
                      uint16_t* out16, double* out64)
{
    double* T = (double*)malloc(65536 * sizeof(double));
    if (!T) return -1;
    build_table(T, dtype);
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < count; ++i) {
        const uint16_t* arow = A + ms[i] * lda;
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const uint16_t b = (layout == OR_LAYOUT_NN) ? B[k * ldb + ns[i]] : B[ns[i] * ldb + k];
            s += T[arow[k]] * T[b];
        }
        if (out64) out64[i] = s;
        if (out16) out16[i] = (dtype == OR_BF16) ? oracle_f64_to_bf16(s) : oracle_f64_to_f16(s);
    }
    free(T);
    return 0;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Batch forms of the codecs, for the exhaustive codec tests. */
void oracle_decode_array(const uint16_t* in, double* out, int64_t n, int dtype)
{
    for (int64_t i = 0; i < n; ++i) {
        if (dtype == OR_E4M3)
            out[i] = oracle_e4m3_to_f64((uint8_t)(in[i] & 0xffu));
        else if (dtype == OR_E5M2)
            out[i] = oracle_e5m2_to_f64((uint8_t)(in[i] & 0xffu));
        else
            out[i] = (dtype == OR_BF16) ? oracle_bf16_to_f64(in[i]) : oracle_f16_to_f64(in[i]);
    }
}

void oracle_encode_array(const double* in, uint16_t* out, int64_t n, int dtype)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = (dtype == OR_BF16) ? oracle_f64_to_bf16(in[i]) : oracle_f64_to_f16(in[i]);
}

/* C = alpha * (A·B) + beta * Cin, the accumulating form of the contraction ("张量缩并：mma
 * 语法" introduces it as C += A × B; alpha = 1, beta = 1 is that form, alpha = 1, beta = 0
 * the plain product).  Same sum as oracle_gemm_rows, then out = alpha * sum + beta * Cin in
 * fp64 and one rounding.  Cin is the logical M x N input, row-major with leading dimension
 * ldcin; with beta == 0 it is not read (may be NULL).  Rows `rows[i]` of the result are
 * written row-major at out16/out64 + i*ldo. */
int oracle_gemm_rows_axpby(const uint16_t* A, const uint16_t* B, const uint16_t* Cin, int64_t N, int64_t K,
                           int64_t lda, int64_t ldb, int64_t ldcin, int layout, int dtype, double alpha,
                           double beta, const int64_t* rows, int64_t nrows, uint16_t* out16, double* out64,
                           int64_t ldo, int nthreads)
{
    double* T = (double*)malloc(65536 * sizeof(double));
    if (!T) return -1;
    build_table(T, dtype);
    int used = 1;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
    {
#pragma omp single
        used = omp_get_num_threads();
        double* acc = (double*)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nrows; ++i) {
            row_f64(T, A, B, rows[i], N, K, lda, ldb, layout, acc);
            for (int64_t n = 0; n < N; ++n) {
                double v = alpha * acc[n];
                if (beta != 0.0) v += beta * T[Cin[rows[i] * ldcin + n]];
                if (out64) out64[i * ldo + n] = v;
                if (out16) out16[i * ldo + n] = (dtype == OR_BF16) ? oracle_f64_to_bf16(v) : oracle_f64_to_f16(v);
            }
        }
        free(acc);
    }
#else
    (void)nthreads;
    double* acc = (double*)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    for (int64_t i = 0; i < nrows; ++i) {
        row_f64(T, A, B, rows[i], N, K, lda, ldb, layout, acc);
        for (int64_t n = 0; n < N; ++n) {
            double v = alpha * acc[n];
            if (beta != 0.0) v += beta * T[Cin[rows[i] * ldcin + n]];
            if (out64) out64[i * ldo + n] = v;
            if (out16) out16[i * ldo + n] = (dtype == OR_BF16) ? oracle_f64_to_bf16(v) : oracle_f64_to_f16(v);
        }
    }
    free(acc);
#endif
    free(T);
    return used;
}

/* C = alpha * (A·B) + beta * Cin with input codes of type in_dtype (f16, bf16, or an 8-bit
 * format whose codes are passed widened to 16 bits) and output / Cin of type out_dtype
 * (f16 or bf16).  The 8-bit contraction with scales ("张量缩并：mma 语法": each result is
 * scaled by sc_a and sc_b after the contraction) is alpha = sc_a * sc_b (* a user alpha). */
int oracle_gemm_rows_typed(const uint16_t* A, const uint16_t* B, const uint16_t* Cin, int64_t N, int64_t K,
                           int64_t lda, int64_t ldb, int64_t ldcin, int layout, int in_dtype, int out_dtype,
                           double alpha, double beta, const int64_t* rows, int64_t nrows, uint16_t* out16,
                           double* out64, int64_t ldo, int nthreads)
{
    double* T = (double*)malloc(65536 * sizeof(double));
    double* TC = (double*)malloc(65536 * sizeof(double));
    if (!T || !TC) {
        free(T);
        free(TC);
        return -1;
    }
    build_table(T, in_dtype);
    build_table(TC, out_dtype);
    int used = 1;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
    {
#pragma omp single
        used = omp_get_num_threads();
#else
    (void)nthreads;
    {
#endif
        double* acc = (double*)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t i = 0; i < nrows; ++i) {
            row_f64(T, A, B, rows[i], N, K, lda, ldb, layout, acc);
            for (int64_t n = 0; n < N; ++n) {
                double v = alpha * acc[n];
                if (beta != 0.0) v += beta * TC[Cin[rows[i] * ldcin + n]];
                if (out64) out64[i * ldo + n] = v;
                if (out16)
                    out16[i * ldo + n] = (out_dtype == OR_BF16) ? oracle_f64_to_bf16(v) : oracle_f64_to_f16(v);
            }
        }
        free(acc);
    }
    free(T);
    free(TC);
    return used;
}

/* ------------------------------------------------------- block-scaled 8-bit operands */

/* Value of an 8-bit scale exponent (the E8M0 format of the OCP microscaling formats:
 * 2^(e - 127), e = 255 is NaN). */
double oracle_e8m0_to_f64(uint8_t e)
{
    return e == 255u ? NAN : ldexp(1.0, (int)e - 127);
}

/* C = alpha * acc + beta * Cin with per-tile scales on 8-bit operands ("张量缩并：mma 语法",
 * quantised operands with per-tile scaling: the contraction of a tile of A with a tile of B
 * is multiplied by the A tile's scale sc_a and the B tile's scale sc_b, and the scaled
 * results are accumulated).  Tiles are 32 long along K and one row (A) or one column (B)
 * wide: sa[m * ldsa + j] scales A[m, 32j .. 32j+31] and sb[n * ldsb + j] scales
 * Beff[32j .. 32j+31, n], both E8M0 exponents.  Per output element, in this order:
 *     part_j = sum_{k in block j} A[m,k] * Beff[k,n]             (the tile contraction)
 *     acc    = sum_j  2^(sa - 127) * 2^(sb - 127) * part_j         (scaled, accumulated)
 * The last block of a K that is not a multiple of 32 holds fewer terms.  Everything in fp64,
 * rounded once to out_dtype.  Same row selection and outputs as oracle_gemm_rows_typed. */
int oracle_gemm_rows_blockscaled(const uint16_t* A, const uint16_t* B, const uint8_t* sa, const uint8_t* sb,
                                 const uint16_t* Cin, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldsa,
                                 int64_t ldsb, int64_t ldcin, int layout, int in_dtype, int out_dtype, double alpha,
                                 double beta, const int64_t* rows, int64_t nrows, uint16_t* out16, double* out64,
                                 int64_t ldo, int nthreads)
{
    const int64_t kBlock = 32;
    double* T = (double*)malloc(65536 * sizeof(double));
    double* TC = (double*)malloc(65536 * sizeof(double));
    if (!T || !TC) {
        free(T);
        free(TC);
        return -1;
    }
    build_table(T, in_dtype);
    build_table(TC, out_dtype);
    const int64_t nblocks = (K + kBlock - 1) / kBlock;
    int used = 1;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
    {
#pragma omp single
        used = omp_get_num_threads();
#else
    (void)nthreads;
    {
#endif
        const size_t n_alloc = (size_t)(N > 0 ? N : 1);
        double* acc = (double*)malloc(n_alloc * sizeof(double));
        double* part = (double*)malloc(n_alloc * sizeof(double));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t i = 0; i < nrows; ++i) {
            const int64_t m = rows[i];
            const uint16_t* arow = A + m * lda;
            for (int64_t n = 0; n < N; ++n) acc[n] = 0.0;
            for (int64_t j = 0; j < nblocks; ++j) {
                const int64_t k0 = j * kBlock, k1 = (k0 + kBlock < K) ? k0 + kBlock : K;
                for (int64_t n = 0; n < N; ++n) part[n] = 0.0;
                for (int64_t k = k0; k < k1; ++k) {
                    const double a = T[arow[k]];
                    for (int64_t n = 0; n < N; ++n)
                        part[n] += a * T[layout == OR_LAYOUT_NN ? B[k * ldb + n] : B[n * ldb + k]];
                }
                const double s_a = oracle_e8m0_to_f64(sa[m * ldsa + j]);
                for (int64_t n = 0; n < N; ++n) acc[n] += s_a * oracle_e8m0_to_f64(sb[n * ldsb + j]) * part[n];
            }
            for (int64_t n = 0; n < N; ++n) {
                double v = alpha * acc[n];
                if (beta != 0.0) v += beta * TC[Cin[m * ldcin + n]];
                if (out64) out64[i * ldo + n] = v;
                if (out16)
                    out16[i * ldo + n] = (out_dtype == OR_BF16) ? oracle_f64_to_bf16(v) : oracle_f64_to_f16(v);
            }
        }
        free(acc);
        free(part);
    }
    free(T);
    free(TC);
    return used;
}

/* ------------------------------------------------------------- 2:4 structured sparsity */

/* "张量缩并：mma 语法", structured sparsity: when at most two of every four consecutive
 * elements along K of a row of A are non-zero, A is kept as its two chosen values per group
 * (Ac, M x K/2) plus metadata naming their positions, and the sparse contraction
 * (mma.row.row.sp with the metadata operand me) multiplies each kept value by the B row it
 * came from.  Metadata words: E[m * lde + j] holds groups 8j .. 8j+7 of row m, group g in
 * bits 4(g - 8j) .. 4(g - 8j) + 3: the low two bits are the position (0..3) of the first kept
 * element, the high two bits that of the second, first < second.
 *
 * Compression of a dense A (M x K, K a multiple of 4): per group the first two non-zero
 * elements are kept (a code is zero when all bits but the sign are 0); when there are fewer,
 * the lowest positions not yet taken complete the pair, and the pair is put in ascending
 * order.  Returns the number of groups with more than two non-zeros (their first two are
 * kept), 0 for a valid 2:4 matrix.  Row padding of Ac / E is not written. */
int64_t oracle_sparse24_compress(const uint16_t* A, int64_t M, int64_t K, int64_t lda, uint16_t* Ac, int64_t ldac,
                                 uint32_t* E, int64_t lde)
{
    int64_t bad = 0;
    const int64_t groups = K / 4;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t j = 0; j * 8 < groups; ++j) E[m * lde + j] = 0u;
        for (int64_t g = 0; g < groups; ++g) {
            const uint16_t* a = A + m * lda + 4 * g;
            int pos[2], n = 0, nonzero = 0;
            for (int i = 0; i < 4; ++i)
                if ((a[i] & 0x7fffu) != 0u) {
                    ++nonzero;
                    if (n < 2) pos[n++] = i;
                }
            if (nonzero > 2) ++bad;
            for (int i = 0; n < 2 && i < 4; ++i)
                if (n == 0 || pos[0] != i) pos[n++] = i;
            if (pos[0] > pos[1]) {
                const int t = pos[0];
                pos[0] = pos[1];
                pos[1] = t;
            }
            Ac[m * ldac + 2 * g] = a[pos[0]];
            Ac[m * ldac + 2 * g + 1] = a[pos[1]];
            E[m * lde + g / 8] |= (uint32_t)(pos[0] | (pos[1] << 2)) << (4 * (g % 8));
        }
    }
    return bad;
}

/* The sparse contraction, as the metadata defines it:
 *     C[m,n] = alpha * sum_g sum_{t<2} Ac[m, 2g+t] * Beff[4g + pos_t(m,g), n] + beta * Cin[m,n]
 * with pos_t read from E as above (K a multiple of 4, K/4 groups), summed in fp64 and rounded
 * once.  Same row selection and outputs as oracle_gemm_rows_typed (16-bit operands). */
int oracle_gemm_rows_sparse24(const uint16_t* Ac, const uint32_t* E, const uint16_t* B, const uint16_t* Cin,
                              int64_t N, int64_t K, int64_t ldac, int64_t lde, int64_t ldb, int64_t ldcin, int layout,
                              int dtype, double alpha, double beta, const int64_t* rows, int64_t nrows,
                              uint16_t* out16, double* out64, int64_t ldo, int nthreads)
{
    double* T = (double*)malloc(65536 * sizeof(double));
    if (!T) return -1;
    build_table(T, dtype);
    const int64_t groups = K / 4;
    int used = 1;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
    {
#pragma omp single
        used = omp_get_num_threads();
#else
    (void)nthreads;
    {
#endif
        double* acc = (double*)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t i = 0; i < nrows; ++i) {
            const int64_t m = rows[i];
            for (int64_t n = 0; n < N; ++n) acc[n] = 0.0;
            for (int64_t g = 0; g < groups; ++g) {
                const uint32_t nib = (E[m * lde + g / 8] >> (4 * (g % 8))) & 0xfu;
                for (int t = 0; t < 2; ++t) {
                    const int64_t k = 4 * g + ((nib >> (2 * t)) & 3u);
                    const double a = T[Ac[m * ldac + 2 * g + t]];
                    for (int64_t n = 0; n < N; ++n)
                        acc[n] += a * T[layout == OR_LAYOUT_NN ? B[k * ldb + n] : B[n * ldb + k]];
                }
            }
            for (int64_t n = 0; n < N; ++n) {
                double v = alpha * acc[n];
                if (beta != 0.0) v += beta * T[Cin[m * ldcin + n]];
                if (out64) out64[i * ldo + n] = v;
                if (out16) out16[i * ldo + n] = (dtype == OR_BF16) ? oracle_f64_to_bf16(v) : oracle_f64_to_f16(v);
            }
        }
        free(acc);
    }
    free(T);
    return used;
}

/*
 * A C program that uses the library the way a C caller would: only include/gemm.h and
 * libdtgemm.so, no Python, no torch, no CUDA headers.
 *
 *   gemm_c_consumer host   host-side entry points (argument checks, the tile map, layout
 *                          sizes, status strings, handle creation on a missing device)
 *   gemm_c_consumer gpu    the above, then GEMMs on host buffers through gemm_run_host on
 *                          device 0 in every configuration, both layouts and both 16-bit
 *                          types, compared bit for bit with the CPU oracle (linked from
 *                          oracle/gemm_oracle.c) on integer inputs in {-2..2}, whose sums
 *                          are exact in fp32 ("NineToothed GEMM 语法入门" §6: one rounding
 *                          on write-back), with guard columns of C that must stay untouched
 *                          (§5: writes outside M x N are dropped)
 *
 * Exit status 0 when every check passes; the first failing check is printed.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "gemm.h"

/* The oracle's entry point (oracle/gemm_oracle.c): rows of C as rounded 16-bit codes. */
int oracle_gemm_rows(const uint16_t* A, const uint16_t* B, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                     int layout, int dtype, const int64_t* rows, int64_t nrows, uint16_t* out16, double* out64,
                     int64_t ldo, int nthreads);
uint16_t oracle_f64_to_f16(double x);
uint16_t oracle_f64_to_bf16(double x);

static int failures = 0;
#define CHECK(cond, ...)                                   \
    do {                                                   \
        if (!(cond)) {                                     \
            fprintf(stderr, "FAIL %s:%d: ", __FILE__, __LINE__); \
            fprintf(stderr, __VA_ARGS__);                  \
            fprintf(stderr, "\n");                         \
            ++failures;                                    \
        }                                                  \
    } while (0)

static void host_checks(void)
{
    static _Alignas(16) uint16_t buf[64 * 64 + 16];
    const void* p = buf;                                  /* 16-byte aligned */
    const char* q = (const char*)buf + 2;                 /* misaligned */
    CHECK(gemm_api_version() == GEMM_API_VERSION, "api version %d", gemm_api_version());
    CHECK(gemm_check_args(p, p, p, 8, 8, 8, 8, 8, 8, GEMM_LAYOUT_NN, GEMM_DTYPE_F16) == GEMM_OK, "valid args");
    CHECK(gemm_check_args(NULL, p, p, 8, 8, 8, 8, 8, 8, GEMM_LAYOUT_NN, GEMM_DTYPE_F16) == GEMM_ERR_INVALID_ARG,
          "null A");
    CHECK(gemm_check_args(p, p, p, -1, 8, 8, 8, 8, 8, GEMM_LAYOUT_NN, GEMM_DTYPE_F16) == GEMM_ERR_INVALID_ARG,
          "negative M");
    CHECK(gemm_check_args(p, p, p, 8, 16, 8, 8, 8, 16, GEMM_LAYOUT_NN, GEMM_DTYPE_F16) == GEMM_ERR_INVALID_ARG,
          "NN ldb < N");
    CHECK(gemm_check_args(p, p, p, 8, 16, 8, 8, 8, 16, GEMM_LAYOUT_TN, GEMM_DTYPE_F16) == GEMM_OK, "TN ldb >= K");
    CHECK(gemm_check_args(q, p, p, 8, 8, 8, 8, 8, 8, GEMM_LAYOUT_NN, GEMM_DTYPE_F16) == GEMM_ERR_UNSUPPORTED,
          "misaligned A");
    CHECK(gemm_check_args(p, p, p, 8, 8, 8, 12, 8, 8, GEMM_LAYOUT_NN, GEMM_DTYPE_F16) == GEMM_ERR_UNSUPPORTED,
          "lda not a multiple of 8");
    CHECK(gemm_check_args(p, p, p, 0, 8, 8, 8, 8, 8, GEMM_LAYOUT_NN, GEMM_DTYPE_F16) == GEMM_OK, "M = 0 is a no-op");
    CHECK(gemm_check_args(p, p, p, 8, 8, 8, 8, 8, 8, 7, GEMM_DTYPE_F16) == GEMM_ERR_INVALID_ARG, "bad layout");
    CHECK(gemm_check_args(p, p, p, 8, 8, 8, 8, 8, 8, GEMM_LAYOUT_NN, 9) == GEMM_ERR_INVALID_ARG, "bad dtype");

    /* The tile map is a bijection of every grid onto itself. */
    for (int64_t tm = 1; tm <= 9; ++tm)
        for (int64_t tn = 1; tn <= 7; ++tn)
            for (int64_t g = 1; g <= 10; g += 3) {
                static unsigned char seen[9 * 7];
                memset(seen, 0, sizeof(seen));
                for (int64_t t = 0; t < tm * tn; ++t) {
                    int64_t r = -1, c = -1;
                    CHECK(gemm_tile_coord(t, tm, tn, g, &r, &c) == GEMM_OK, "tile_coord status");
                    CHECK(r >= 0 && r < tm && c >= 0 && c < tn, "tile %lld outside the grid", (long long)t);
                    if (r >= 0 && r < tm && c >= 0 && c < tn) {
                        CHECK(!seen[r * tn + c], "tile (%lld, %lld) twice", (long long)r, (long long)c);
                        seen[r * tn + c] = 1;
                    }
                }
            }
    int64_t r, c;
    CHECK(gemm_tile_coord(6, 2, 3, 1, &r, &c) == GEMM_ERR_INVALID_ARG, "tile past the grid");

    /* Side-data sizes from their definitions in gemm.h. */
    CHECK(gemm_sp_meta_bytes(128, 64) == 4096, "one metadata chunk");
    CHECK(gemm_sp_meta_bytes(129, 65) == 4 * 4096, "ragged metadata chunks");
    CHECK(gemm_sp_meta_bytes(0, 64) == 0, "no metadata");
    CHECK(gemm_mx_scale_bytes(128, 128) == 512, "one scale chunk");
    CHECK(gemm_mx_scale_bytes(300, 520) == 3 * 5 * 512, "ragged scale chunks");

    for (int s = GEMM_OK; s <= GEMM_ERR_TIMEOUT + 1; ++s)
        CHECK(gemm_status_string(s) != NULL && gemm_status_string(s)[0] != '\0', "status string %d", s);
    CHECK(gemm_create(NULL, 0) == GEMM_ERR_INVALID_ARG, "create without an out pointer");
    gemm_handle_t none = NULL;
    const gemm_status_t st = gemm_create(&none, 9999);
    CHECK(st != GEMM_OK && none == NULL, "create on a missing device: %d", st);
    CHECK(gemm_destroy(NULL) == GEMM_OK, "destroy NULL");
    /* Struct sizes as a C compiler lays them out (the Python binding checks against these). */
    printf("sizeof gemm_plan_t %zu gemm_args_t %zu\n", sizeof(gemm_plan_t), sizeof(gemm_args_t));
}

/* Deterministic integers in {-2..2}, as 16-bit codes of the type. */
static uint16_t int_code(uint32_t* state, int dtype)
{
    *state = *state * 1664525u + 1013904223u;
    const int v = (int)((*state >> 16) % 5u) - 2;
    return dtype == GEMM_DTYPE_BF16 ? oracle_f64_to_bf16((double)v) : oracle_f64_to_f16((double)v);
}

static void gpu_checks(void)
{
    gemm_handle_t h = NULL;
    gemm_status_t st = gemm_create(&h, 0);
    CHECK(st == GEMM_OK, "gemm_create: %s", gemm_status_string(st));
    if (st != GEMM_OK) return;
    const int64_t shapes[][3] = {{300, 200, 130}, {1000, 700, 515}, {65, 97, 130}, {1, 1, 1}};
    const int configs[] = {GEMM_CONFIG_AUTO, GEMM_CONFIG_128x256, GEMM_CONFIG_128x128, GEMM_CONFIG_128x64,
                           GEMM_CONFIG_256x256};
    const uint16_t guard = 0x7777;
    uint32_t state = 12345u;
    for (size_t si = 0; si < sizeof(shapes) / sizeof(shapes[0]); ++si)
        for (int layout = GEMM_LAYOUT_NN; layout <= GEMM_LAYOUT_TN; ++layout)
            for (int dtype = GEMM_DTYPE_F16; dtype <= GEMM_DTYPE_BF16; ++dtype) {
                const int64_t M = shapes[si][0], N = shapes[si][1], K = shapes[si][2];
                const int64_t lda = (K + 7) / 8 * 8 + 8;
                const int64_t brows = layout == GEMM_LAYOUT_NN ? K : N;
                const int64_t bcols = layout == GEMM_LAYOUT_NN ? N : K;
                const int64_t ldb = (bcols + 7) / 8 * 8 + 8;
                const int64_t ldc = (N + 7) / 8 * 8 + 8;
                uint16_t* A = (uint16_t*)malloc((size_t)(M * lda) * 2);
                uint16_t* B = (uint16_t*)malloc((size_t)(brows * ldb) * 2);
                uint16_t* C = (uint16_t*)malloc((size_t)(M * ldc) * 2);
                uint16_t* ref = (uint16_t*)malloc((size_t)(M * N) * 2);
                int64_t* rows = (int64_t*)malloc((size_t)M * sizeof(int64_t));
                if (!A || !B || !C || !ref || !rows) {
                    CHECK(0, "host allocation");
                    return;
                }
                for (int64_t i = 0; i < M * lda; ++i) A[i] = int_code(&state, dtype);
                for (int64_t i = 0; i < brows * ldb; ++i) B[i] = int_code(&state, dtype);
                for (int64_t i = 0; i < M; ++i) rows[i] = i;
                CHECK(oracle_gemm_rows(A, B, N, K, lda, ldb, layout, dtype, rows, M, ref, NULL, N, 0) > 0,
                      "oracle");
                for (size_t ci = 0; ci < sizeof(configs) / sizeof(configs[0]); ++ci) {
                    CHECK(gemm_set_option(h, GEMM_OPT_CONFIG, configs[ci]) == GEMM_OK, "set config");
                    for (int64_t i = 0; i < M * ldc; ++i) C[i] = guard;
                    st = gemm_run_host(h, A, B, C, M, N, K, lda, ldb, ldc, layout, dtype, NULL);
                    CHECK(st == GEMM_OK, "gemm_run_host %lldx%lldx%lld: %s", (long long)M, (long long)N,
                          (long long)K, gemm_status_string(st));
                    int64_t bad = 0, bad_guard = 0;
                    for (int64_t m = 0; m < M; ++m)
                        for (int64_t n = 0; n < ldc; ++n) {
                            if (n < N)
                                bad += C[m * ldc + n] != ref[m * N + n];
                            else
                                bad_guard += C[m * ldc + n] != guard;
                        }
                    CHECK(bad == 0 && bad_guard == 0,
                          "%lldx%lldx%lld layout %d dtype %d config %d: %lld codes differ from the oracle, "
                          "%lld guard codes written",
                          (long long)M, (long long)N, (long long)K, layout, dtype, configs[ci], (long long)bad,
                          (long long)bad_guard);
                }
                free(A);
                free(B);
                free(C);
                free(ref);
                free(rows);
            }
    CHECK(gemm_set_option(h, GEMM_OPT_CONFIG, GEMM_CONFIG_AUTO) == GEMM_OK, "reset config");
    gemm_plan_t plan;
    CHECK(gemm_query_plan(h, 8192, 8192, 8192, GEMM_LAYOUT_TN, GEMM_DTYPE_BF16, &plan) == GEMM_OK &&
              plan.cluster == 2 && plan.bm == 256 && plan.bn == 256 && plan.raster_group == 12 && plan.k_snake == 1,
          "plan of the square 8192^3 problem");
    CHECK(gemm_destroy(h) == GEMM_OK, "destroy");
}

int main(int argc, char** argv)
{
    const int gpu = argc > 1 && strcmp(argv[1], "gpu") == 0;
    host_checks();
    if (gpu) gpu_checks();
    if (failures) {
        fprintf(stderr, "%d check(s) failed\n", failures);
        return 1;
    }
    printf("gemm_c_consumer %s: ok\n", gpu ? "gpu" : "host");
    return 0;
}

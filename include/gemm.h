/*
 * gemm.h -- C ABI of the GB300 (sm_103a) tiled dense GEMM library.
 *
 * Operation (every entry point that computes): C = A·B with 16-bit inputs, an fp32
 * accumulator and a 16-bit output in the input type, rounded to nearest-even once.
 *   - "NineToothed GEMM 语法入门" (NineToothed GEMM syntax primer) §2: the accumulator
 *     starts at zero, each K block adds dot(A tile, B tile), the output is assigned once
 *     (so C is overwritten, alpha = 1, beta = 0); §6: fp32 accumulation, 16-bit storage.
 *   - same page §3: output tile (i, j) covers C[i*BM:, j*BN:] and reads A[i*BM:, p*BK:] and
 *     B[p*BK:, j*BN:] for every K block p; §5: reads past M/N/K count as zero and writes
 *     past M x N are dropped, so any M, N, K >= 0 is accepted.
 *   - "张量缩并：mma 语法" (Croqtile tutorial ch. 4), the one-warp kernel: the kernel
 *     writes its output in place and takes B as [N, K] -- the TN layout below.
 *
 * Layouts.  Every matrix is row-major with a leading dimension (elements between rows):
 *   A: M x K, lda >= K.
 *   GEMM_LAYOUT_NN: B stored K x N, ldb >= N   (C = A · B)
 *   GEMM_LAYOUT_TN: B stored N x K, ldb >= K   (C = A · Bstored^T)
 *   C: M x N, ldc >= N.  Elements of C outside the M x N window (row padding) are never
 *   written; elements of A/B outside their logical window are never read.
 *
 * Alignment (the tensor-memory-access engine needs 16-byte aligned bases and row
 * pitches): A, B, C must be 16-byte aligned and lda, ldb, ldc multiples of 8 elements,
 * otherwise GEMM_ERR_UNSUPPORTED.  There is no fallback path.
 *
 * Ownership.  The caller owns A, B, C and the stream; the handle owns the watchdog's
 * 16-byte error word, a stream-K workspace (fp32 partial sums and arrival counters, about
 * 40 MB on a 152-SM GPU, allocated by gemm_create), a cache of tensor-map descriptors and,
 * after the first gemm_run_host, device staging buffers plus that path's streams and
 * events.  A handle may be used from one host thread at a time, and its launches must not
 * overlap on the GPU (they share the workspace): enqueue them on one stream or order them.
 * Aliasing C with A or B is undefined.
 *
 * Errors.  Every entry point returns a status; nothing throws across the ABI.
 */
#ifndef DTG_GEMM_H
#define DTG_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GEMM_API_VERSION 3

typedef struct gemm_handle_s* gemm_handle_t;

typedef int32_t gemm_layout_t;
enum { GEMM_LAYOUT_NN = 0, GEMM_LAYOUT_TN = 1 };

/* Element types.  F16 and BF16 serve as operand and output types; E4M3 and E5M2 (8-bit
 * floats: 1-4-3 with bias 7 and no infinities, 1-5-2 with bias 15) are operand types only,
 * accepted by gemm_run_ex. */
typedef int32_t gemm_dtype_t;
enum { GEMM_DTYPE_F16 = 0, GEMM_DTYPE_BF16 = 1, GEMM_DTYPE_E4M3 = 2, GEMM_DTYPE_E5M2 = 3 };

typedef int32_t gemm_status_t;
enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1, /* null handle/pointer, negative size, ld too small, bad enum   */
    GEMM_ERR_UNSUPPORTED = 2, /* misaligned base or ld, a dimension >= 2^31                  */
    GEMM_ERR_ARCH = 3,        /* device is not compute capability 10.3 (sm_103)               */
    GEMM_ERR_CUDA = 4,        /* a CUDA runtime/driver call or a launch failed                 */
    GEMM_ERR_TIMEOUT = 5      /* a device-side wait gave up (watchdog); see gemm_error_info   */
};

/* Tunables and test hooks for gemm_set_option / gemm_get_option. */
typedef int32_t gemm_option_t;
enum {
    GEMM_OPT_CONFIG = 0,       /* kernel configuration: GEMM_CONFIG_* (default AUTO)          */
    GEMM_OPT_TIMEOUT_NS = 1,   /* device watchdog limit per wait, ns (default 2e9, min 1e6)   */
    GEMM_OPT_MAX_CTAS = 2,     /* cap on persistent CTAs (0 = one per SM); tests use it to
                                  make each CTA walk several tiles                            */
    GEMM_OPT_RASTER_GROUP = 3, /* output-tile raster: M tiles per group (L2 reuse), >= 1; 0 (the
                                  default) = the tile rows whose A holds about 48 MiB, at most
                                  16 and at most the tile columns (8192^3 bf16: 12; E4M3: 16;
                                  16384 x 1024 x 8192 fp16: 4); gemm_query_plan reports the
                                  value used                                                  */
    GEMM_OPT_FAULT_INJECT = 4, /* test hook: 1 = the first work unit (a CTA, or both CTAs of a
                                  pair) loads one ring stage nowhere and leaves it unarmed, so
                                  a consumer wait runs out and the watchdog path returns
                                  GEMM_ERR_TIMEOUT through gemm_sync_status (no GPU fault)   */
    GEMM_OPT_STREAM_K = 5,     /* 1 (default): when whole tiles would leave the last wave
                                  part-empty (or the whole problem is under one wave), share
                                  the K blocks of the last tiles evenly between CTAs (partial
                                  sums merged in K order, so results are deterministic);
                                  0: whole tiles only ("NineToothed GEMM 语法入门" §4: a K
                                  loop split across programs needs a merge)                  */
    GEMM_OPT_HOST_ROW_CHUNKS = 6, /* gemm_run_host: row chunks of A and C, 1..16 (default 8;
                                  chunks are at least 1024 rows)                              */
    GEMM_OPT_HOST_COL_CHUNKS = 7, /* gemm_run_host: column chunks of C (B's rows for TN, its
                                  columns for NN), 1..8 (default 4; at least 2048 columns)   */
    GEMM_OPT_SK_MIN_BLOCKS = 8, /* shortest stream-K share of a part-empty last wave, in K
                                  blocks (default 8, >= 1)                                  */
    GEMM_OPT_SPLIT_MIN_BLOCKS = 9, /* a problem under one wave (fewer tiles than the CTAs or
                                  pairs that fit) has its K blocks split over more units only
                                  when every share holds at least this many (default 32;
                                  0 = never): the merge costs a few microseconds of dependent
                                  global-memory traffic, which only long K loops repay.  The
                                  units are then as many as shares of that length allow, if
                                  more than the tiles                                         */
    GEMM_OPT_K_SNAKE = 10      /* 1 (default): every second work item of a CTA (or pair) walks
                                  its K blocks from the last down, so that a wave of items
                                  starts on the K slices the wave before read last (still in
                                  L2): bf16 8192^3 ~1 % faster in bursts, ~2 % under the power
                                  limit; 0: every item from the first K block up.  Block-scaled
                                  kernels ignore it.  Changes only the order of the fp32
                                  additions within an item (results stay deterministic)       */
};

typedef int32_t gemm_config_t;
enum {
    GEMM_CONFIG_AUTO = 0,
    GEMM_CONFIG_128x256 = 1,   /* 1-CTA tile 128 x 256 x 64, 4-stage ring                      */
    GEMM_CONFIG_128x128 = 2,   /* 1-CTA tile 128 x 128 x 64, 6-stage ring (more tiles)         */
    GEMM_CONFIG_256x256 = 3,   /* 2-CTA cluster tile 256 x 256 x 64 (cta_group::2)             */
    GEMM_CONFIG_128x64 = 4     /* 1-CTA tile 128 x 64 x 64, 8-stage ring (small problems: more
                                  SMs taking in operands; 8-bit operands run 128 x 128 and
                                  side-data kernels 128 x 256 instead)                       */
};

/* What gemm_run would launch for a problem (for benchmarks and tests). */
typedef struct {
    int32_t config;     /* GEMM_CONFIG_* actually chosen                                     */
    int32_t bm, bn, bk; /* output tile (per cluster) and K block                             */
    int32_t stages;     /* shared-memory ring depth                                          */
    int32_t cluster;    /* CTAs per cluster (1 or 2)                                          */
    int64_t tiles_m, tiles_n, k_blocks;
    int64_t grid;       /* CTAs launched (persistent)                                        */
    int32_t threads;    /* threads per CTA                                                   */
    int32_t smem_bytes; /* dynamic shared memory per CTA                                     */
    int64_t dp_tiles;   /* tiles done whole; the rest are shared out by K blocks (stream-K) */
    int64_t sk_base;    /* stream-K K blocks per work unit (the first sk_extra units: +1)    */
    int64_t sk_extra;
    int64_t raster_group; /* tile rows per group of the raster order the launch uses        */
    int64_t k_snake;      /* 1: every second work item walks its K blocks from the last down
                             (GEMM_OPT_K_SNAKE; always 0 for block-scaled operands)         */
} gemm_plan_t;

/* Create a handle bound to CUDA device `device`.  Checks that the device is sm_103,
 * reads its SM count and allocates the device error word and the stream-K workspace.
 * Returns INVALID_ARG (out == NULL or no such device), ARCH, or CUDA. */
gemm_status_t gemm_create(gemm_handle_t* out, int device);

/* Free everything the handle owns.  Synchronises the device first.  NULL is accepted. */
gemm_status_t gemm_destroy(gemm_handle_t h);

/* Enqueue C = A·B on `stream` (a cudaStream_t; NULL = legacy default stream) and return
 * without waiting.  A, B, C are device pointers.  M == 0 or N == 0 is a no-op; K == 0
 * writes zeros to C (the empty sum).  Device-side watchdog expiries are reported later
 * by gemm_sync_status.  Launch failures return GEMM_ERR_CUDA. */
gemm_status_t gemm_run(gemm_handle_t h, const void* A, const void* B, void* C,
                       int64_t M, int64_t N, int64_t K,
                       int64_t lda, int64_t ldb, int64_t ldc,
                       gemm_layout_t layout, gemm_dtype_t dtype, void* stream);

/* The general form: C = alpha * scale_a * scale_b * A·B + beta * C, with C stored row-major
 * or column-major and 16-bit or 8-bit operands.
 *   - "张量缩并：mma 语法" states the contraction as C += A × B (alpha = beta = 1); its
 *     transposed store (mma.store.transp) writes the result with rows and columns swapped,
 *     which is c_col_major here; its scaled form (mma.row.row.scale with sc_a, sc_b) scales
 *     each result after the contraction, which is scale_a, scale_b here (per-tensor scales,
 *     the usual companions of 8-bit operands).
 *   - dtype: operand type of A and B (F16, BF16, E4M3 or E5M2).  out_dtype: type of C (F16
 *     or BF16); for 16-bit operands it must equal dtype.
 *   - alpha, beta, scale_a, scale_b: finite fp32 scalars.  The result is
 *     (alpha * scale_a * scale_b) * acc + beta * C_old in fp32 (the three factors multiplied
 *     in fp32 first), rounded once to out_dtype.  With beta == 0, C is not read (it may hold
 *     anything, NaN included).  K == 0 gives C = beta * C.
 *   - c_col_major = 0: C[m, n] at C + m * ldc + n (ldc >= N), as in gemm_run.
 *     c_col_major = 1: C[m, n] at C + n * ldc + m (ldc >= M; C stored N x M row-major).
 *   - 8-bit operands: lda and ldb must be multiples of 16 elements (16 bytes); otherwise
 *     A, B, layouts, alignment rules and status codes are those of gemm_run.
 * alpha = scale_a = scale_b = 1, beta = 0, c_col_major = 0, out_dtype = dtype is exactly
 * gemm_run. */
typedef struct {
    const void* A;
    const void* B;
    void* C;
    int64_t M, N, K;
    int64_t lda, ldb, ldc;
    gemm_layout_t layout;
    gemm_dtype_t dtype;
    float alpha;
    float beta;
    int32_t c_col_major;
    gemm_dtype_t out_dtype;
    float scale_a;
    float scale_b;
} gemm_args_t;

gemm_status_t gemm_run_ex(gemm_handle_t h, const gemm_args_t* args, void* stream);

/* 8-bit operands with per-tile scales: C = alpha * scale_a * scale_b * acc + beta * C with
 *     acc[m, n] = sum_j 2^(ea[m, j] - 127) * 2^(eb[n, j] - 127) * sum_{k in block j} A[m, k] * Beff[k, n]
 * over K blocks j of 32 elements (the last one shorter when K % 32 != 0).  This is the scaled
 * contraction of "张量缩并：mma 语法" (each tile's product multiplied by the A tile's scale
 * sc_a and the B tile's scale sc_b), with tiles of one row of A, or one column of B, by 32
 * K elements, and scales in E8M0 (8-bit exponents; 255 is NaN): tcgen05's block-scaled MMA
 * applies them inside the contraction, so no separate dequantisation pass runs.
 *   - args: as for gemm_run_ex, with dtype E4M3 or E5M2 (anything else: INVALID_ARG).
 *     Configurations: the 256 x 256 CTA pair where gemm_run would take a pair tile (at least
 *     one pair tile per pair of SMs), else the one-CTA 128 x 256 tile; GEMM_OPT_CONFIG may ask
 *     for either (GEMM_CONFIG_256x256: the pair; _128x256 / _128x128: one CTA).
 *   - sfa: the exponents ea of A (M x ceil(K/32)), sfb: those of B (one row per column n of
 *     Beff, N x ceil(K/32)), both device pointers, 16-byte aligned, in the chunked layout that
 *     gemm_mx_pack_scales writes (gemm_mx_scale_bytes(M, K) and (N, K) bytes).  Unused when
 *     K == 0; otherwise null is INVALID_ARG and misalignment UNSUPPORTED.
 *   - Padding entries of the chunked layout must hold finite scales (the packer writes 127). */
gemm_status_t gemm_run_mx(gemm_handle_t h, const gemm_args_t* args, const void* sfa, const void* sfb,
                          void* stream);

/* 2:4 structured sparsity ("张量缩并：mma 语法", structured sparsity: with at most two
 * non-zeros in every four consecutive elements along K of a row of A, the hardware skips the
 * zero products; a metadata operand names the kept elements).  C = alpha * scale_a * scale_b *
 * A·B + beta * C where A is given compressed:
 *   - args->A: the kept values, M x K/2 (lda >= K/2, a multiple of 8; 16-byte aligned): for
 *     every group g of four along K, the two kept elements in ascending position order.
 *   - meta: their positions, in the chunked layout gemm_sp_compress writes
 *     (gemm_sp_meta_bytes(M, K) bytes, 16-byte aligned): chunk (row block rb of 128 rows,
 *     K stage s of 64) starts at byte (rb * ceil(K/64) + s) * 4096 and has two 2048-byte
 *     halves, for K [64 s, 64 s + 32) and [64 s + 32, 64 s + 64); in a half, lane l of the
 *     block takes 16 bytes at l * 16: a 32-bit word, then three words of padding.  A group
 *     of four K elements takes 4 bits: the low two give the position (0..3) of the first kept
 *     element, the high two the second, first < second.  Rows pair up: for rows r = 16 b + i
 *     and r + 8 (i < 8), lane r's word holds groups 0-3 of the half's 32 K of row r (bits
 *     0-15, group q at bits 4q) and of row r + 8 (bits 16-31); lane r + 8's word holds
 *     groups 4-7 of the two rows the same way.  Positions must be distinct and ascending
 *     (the pattern of padding rows and groups is (0, 1)); otherwise the result is undefined.
 *   - dtype F16 or BF16 with out_dtype == dtype; K a multiple of 4 (else UNSUPPORTED); B, C,
 *     alpha, beta, c_col_major and the status codes as in gemm_run_ex.  K == 0 gives C = beta
 *     * C and ignores meta.  Configurations: the CTA pair where gemm_run would take it, else
 *     the one-CTA 128 x 256 tile; GEMM_OPT_CONFIG may ask for either. */
gemm_status_t gemm_run_sp(gemm_handle_t h, const gemm_args_t* args, const void* meta, void* stream);

/* Bytes of the chunked sparsity metadata for M rows and K: ceil(M/128) * ceil(K/64) * 4096
 * (0 when M or K is 0). */
int64_t gemm_sp_meta_bytes(int64_t M, int64_t K);

/* Enqueue on `stream` the compression of a dense 2:4 matrix A (M x K, lda >= K, device, 16-bit
 * dtype F16 or BF16) into Ac (M x K/2, ldac >= K/2) and meta (gemm_sp_meta_bytes(M, K) bytes,
 * 16-byte aligned).  Per group of four along K the first two non-zero elements are kept (a
 * value is zero when it is +0 or -0); fewer are completed with the lowest free positions, in
 * ascending order.  Groups with more than two non-zeros keep their first two and are counted
 * into *bad_groups (a device int32, added to atomically; may be NULL).  M == 0 or K == 0 is a
 * no-op; K % 4 != 0 or a misaligned meta is UNSUPPORTED; null pointers, lda < K or
 * ldac < K/2 are INVALID_ARG. */
gemm_status_t gemm_sp_compress(gemm_handle_t h, const void* A, int64_t M, int64_t K, int64_t lda, gemm_dtype_t dtype,
                               void* Ac, int64_t ldac, void* meta, int32_t* bad_groups, void* stream);

/* Bytes of the chunked block-scale layout for `rows` rows and K elements of K:
 * ceil(rows / 128) * ceil(K / 128) * 512 (0 when rows or K is 0).  Chunk (rb, g) covers rows
 * [128 rb, 128 rb + 128) and K blocks [4 g, 4 g + 4) and starts at byte (rb * ceil(K/128) + g)
 * * 512; inside it, row r and K block c of the chunk sit at byte (r % 32) * 16 + (r / 32) * 4
 * + c. */
int64_t gemm_mx_scale_bytes(int64_t rows, int64_t K);

/* Enqueue on `stream` the rearrangement of row-major exponents src[r * ld + j] (rows x
 * kblocks bytes, ld >= kblocks; device memory) into the chunked layout at dst (device,
 * gemm_mx_scale_bytes(rows, 32 * kblocks) bytes), padding with 127 (a scale of 1).
 * rows == 0 or kblocks == 0 is a no-op; negative sizes, null pointers or ld < kblocks are
 * INVALID_ARG. */
gemm_status_t gemm_mx_pack_scales(gemm_handle_t h, const void* src, int64_t rows, int64_t kblocks, int64_t ld,
                                  void* dst, void* stream);

/* Same operation on HOST buffers (pinned memory lets the copies run as DMA): copies A and
 * B to handle-owned device buffers, runs the kernel, copies C back (only the M x N window,
 * never the row padding) and synchronises `stream`.  The copies and the GEMMs overlap: A
 * and C are cut into row chunks and C's columns into column chunks (GEMM_OPT_HOST_ROW_CHUNKS,
 * GEMM_OPT_HOST_COL_CHUNKS); the inputs go over in order on one internal stream, each block
 * of C is computed on `stream` as soon as its rows of A and columns of B are in and goes
 * back on another internal stream while later inputs arrive.  Returns the watchdog status
 * as gemm_sync_status does.  Grows its device buffers on demand (cudaMalloc) -- call once
 * outside any timed region to size them. */
gemm_status_t gemm_run_host(gemm_handle_t h, const void* A, const void* B, void* C,
                            int64_t M, int64_t N, int64_t K,
                            int64_t lda, int64_t ldb, int64_t ldc,
                            gemm_layout_t layout, gemm_dtype_t dtype, void* stream);

/* Synchronise `stream`, then read and clear the device error word.  Returns
 * GEMM_ERR_TIMEOUT if any kernel launched through this handle since the last call hit
 * its watchdog, GEMM_ERR_CUDA if the stream reports an error, else GEMM_OK. */
gemm_status_t gemm_sync_status(gemm_handle_t h, void* stream);

/* Details of the last watchdog expiry seen by gemm_sync_status / gemm_run_host:
 * info[0] = 1 (timeout), info[1] = role (0 producer, 1 mma, 2 epilogue, 3 drain, 4 side-data copies),
 * info[2] = CTA index, info[3] = tile index * 65536 + K block.  Zeros if none. */
gemm_status_t gemm_error_info(gemm_handle_t h, int32_t info[4]);

gemm_status_t gemm_set_option(gemm_handle_t h, gemm_option_t opt, int64_t value);
gemm_status_t gemm_get_option(gemm_handle_t h, gemm_option_t opt, int64_t* value);

/* Fill *plan with the launch gemm_run would make for this problem (no GPU work). */
gemm_status_t gemm_query_plan(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                              gemm_layout_t layout, gemm_dtype_t dtype, gemm_plan_t* plan);

/* Operand kinds for gemm_query_plan_kind: the operands of gemm_run / gemm_run_ex (dense), of
 * gemm_run_mx (8-bit with E8M0 block scales) and of gemm_run_sp (a 2:4-sparse A). */
typedef int32_t gemm_kind_t;
enum { GEMM_KIND_DENSE = 0, GEMM_KIND_BLOCK_SCALED = 1, GEMM_KIND_SPARSE24 = 2 };

/* Fill *plan with the launch the entry point for operands of `kind` would make (no GPU
 * work).  dtype is the operand type: F16/BF16/E4M3/E5M2 for DENSE (the same as
 * gemm_query_plan), E4M3/E5M2 for BLOCK_SCALED, F16/BF16 for SPARSE24 (K is the logical,
 * uncompressed K).  INVALID_ARG for another combination. */
gemm_status_t gemm_query_plan_kind(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                                   gemm_layout_t layout, gemm_dtype_t dtype, gemm_kind_t kind,
                                   gemm_plan_t* plan);

/* The argument checks gemm_run applies, without a handle or a GPU: INVALID_ARG,
 * UNSUPPORTED or OK exactly as gemm_run would return them before launching.  Pointers
 * are only inspected (null, alignment), never dereferenced. */
gemm_status_t gemm_check_args(const void* A, const void* B, const void* C,
                              int64_t M, int64_t N, int64_t K,
                              int64_t lda, int64_t ldb, int64_t ldc,
                              gemm_layout_t layout, gemm_dtype_t dtype);

/* Host copy of the device tile scheduler's map: linear tile index -> (tile row, tile
 * column) for a tiles_m x tiles_n grid rastered in groups of `group_m` tile rows.
 * Pure function, needs no GPU (tests check it is a bijection).  Returns INVALID_ARG if
 * tile is out of range or an argument is not positive. */
gemm_status_t gemm_tile_coord(int64_t tile, int64_t tiles_m, int64_t tiles_n, int64_t group_m,
                              int64_t* tile_m, int64_t* tile_n);

/* C = A·B without a handle and without allocating any device memory.
 *
 * None of the source pages has a counterpart to this entry point; it exists for callers that cannot
 * call cudaMalloc: plug-ins running inside an engine that owns every byte of device
 * memory through its own pool, latency-critical paths that cannot afford the implicit device-wide
 * synchronisation an allocation may cause, or a process already at its memory limit.
 *
 * Arguments and layouts are those of gemm_run (A, B, C device pointers; same checks and
 * status codes), and so are the kernel and its tile configuration; the schedule takes whole
 * tiles only (gemm_run may split the K blocks of a last, part-empty wave between CTAs), so
 * the fp32 sums may run in another order: results agree within rounding, bit for bit on
 * integer-valued inputs.  The only
 * scratch the kernel needs -- its 16-byte watchdog record -- lives in a 256-byte
 * file-scope __device__ array inside the library (every GPU that loads the library keeps
 * those 256 bytes until the process exits).  A call whose scratch need exceeded that
 * maximum would be rejected with GEMM_ERR_UNSUPPORTED; this kernel's need is fixed at
 * 16 bytes, so no problem size is rejected for that reason.
 *
 * Set-up: the first call on a device (the caller's current device) looks up the array's
 * device address with cudaGetSymbolAddress and checks the device is sm_103; make that
 * first call before any stream capture.  Every call clears the record with
 * cudaMemsetAsync on `stream`, then launches.  All calls share the one record, so calls
 * that overlap on the GPU (different streams, no ordering) race on it.
 *
 * watchdog_info: NULL -> the call returns as soon as the work is enqueued (asynchronous,
 * like gemm_run) and a watchdog expiry is not reported.  Non-NULL (host memory, 4 int32)
 * -> the call synchronises `stream`, copies the record there ({1, role, CTA, tile*65536 +
 * K block} after an expiry, zeros otherwise) and returns GEMM_ERR_TIMEOUT on an expiry. */
gemm_status_t gemm_run_noalloc(const void* A, const void* B, void* C,
                               int64_t M, int64_t N, int64_t K,
                               int64_t lda, int64_t ldb, int64_t ldc,
                               gemm_layout_t layout, gemm_dtype_t dtype, void* stream,
                               int32_t* watchdog_info);

/* Static description of a status code.  Never NULL. */
const char* gemm_status_string(gemm_status_t s);

/* GEMM_API_VERSION of the built library. */
int32_t gemm_api_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DTG_GEMM_H */

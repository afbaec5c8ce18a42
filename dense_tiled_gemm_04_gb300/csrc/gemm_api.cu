// Host side of the C ABI declared in include/gemm.h: argument validation, TMA tensor-map
// encoding, the choice of kernel configuration and the launch.  All arithmetic runs in
// the kernels of gemm_kernel.cuh.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "gemm.h"
#include "kernel_set.cuh"

namespace {

using dtg::KernelChoice;
using dtg::KernelParams;

constexpr int64_t kGroupPanelBytes = 48ll << 20;  // automatic raster group: A bytes of a group's tile rows
constexpr int64_t kMaxAutoGroup = 16;             // and at most this many tile rows
constexpr int64_t kTimeoutDefaultNs = 2000000000LL;  // 2 s per wait
constexpr int kTmapCacheMax = 64;
constexpr int32_t kTmapBytes = -1;  // get_tmap element type: raw bytes (side data)
constexpr int kNumSlots = 96;  // 4 configurations x 12 operand/output types x 2 layouts
constexpr int64_t kMinStreamKBlocks = 8;   // default shortest stream-K share (GEMM_OPT_SK_MIN_BLOCKS)
constexpr int64_t kMinSplitBlocks = 32;    // default shortest share of a split under one wave (GEMM_OPT_SPLIT_MIN_BLOCKS)

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool load_encode_fn()
{
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

struct TmapKey {
    const void* ptr;
    uint64_t inner, outer, pitch_bytes;
    uint32_t box_inner, box_outer;
    int32_t dtype;
    int32_t swizzle;
    bool operator==(const TmapKey& o) const
    {
        return ptr == o.ptr && inner == o.inner && outer == o.outer && pitch_bytes == o.pitch_bytes &&
               box_inner == o.box_inner && box_outer == o.box_outer && dtype == o.dtype && swizzle == o.swizzle;
    }
};

// Epilogue of a launch: C = alpha * A·B + beta * C, C row-major or column-major, of
// type `out` (< 0: the operand type).
struct Epilogue {
    float alpha = 1.0f;
    float beta = 0.0f;
    int32_t col_major = 0;
    gemm_dtype_t out = -1;
    const void* sfa = nullptr;  // block scales (8-bit operands): both set, or both null
    const void* sfb = nullptr;
    const void* meta = nullptr;  // 2:4 sparsity metadata: A is the compressed (M x K/2) matrix
};

struct TmapEntry {
    TmapKey key;
    CUtensorMap map;
};

// Tunables a launch reads (a handle's options, or the defaults).
struct LaunchOptions {
    int64_t config = GEMM_CONFIG_AUTO;
    int64_t timeout_ns = kTimeoutDefaultNs;
    int64_t max_ctas = 0;
    int64_t raster_group = 0;  // 0: automatic
    int64_t fault_inject = 0;
    int64_t stream_k = 1;
    int64_t sk_min_blocks = kMinStreamKBlocks;
    int64_t split_min_blocks = kMinSplitBlocks;
    int64_t k_snake = 1;
    int64_t host_row_chunks = 8;
    int64_t host_col_chunks = 4;
};

// Per-device facts and lazily-set per-kernel state.  Guarded by `mu`.
struct DeviceState {
    int num_sms = 0;
    std::mutex mu;
    bool attrs_set[kNumSlots] = {};
    int max_clusters[kNumSlots] = {};  // pair kernels: co-resident clusters (0 = not yet queried)
};

// Streams and events of gemm_run_host's copy/compute pipeline (created on first use).
struct HostPipe {
    static constexpr int kMaxRowChunks = 16;  // row chunks of A (and C)
    static constexpr int kMaxColChunks = 8;   // column chunks of C (B's rows for TN, columns for NN)
    static constexpr int kMaxPieces = kMaxRowChunks + kMaxColChunks;
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;  // host -> device copies, in order; device -> host copies
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t arrived[kMaxPieces] = {};      // per input piece, in transfer order
    cudaEvent_t computed[kMaxPieces] = {};     // per GEMM launch
};

// Stream-K workspace: fp32 partial sums and arrival counters (see gemm_kernel.cuh).
struct Workspace {
    float* partials = nullptr;
    int32_t* counters = nullptr;
    size_t partial_floats = 0;  // capacity
    int64_t counter_count = 0;  // capacity
};

}  // namespace

struct gemm_handle_s {
    int device = 0;
    int32_t* d_err = nullptr;  // 4 ints
    int32_t last_info[4] = {0, 0, 0, 0};
    LaunchOptions opts;
    DeviceState dev;
    Workspace ws;
    std::vector<TmapEntry> tmaps;
    // gemm_run_host staging and pipeline
    void* d_stage = nullptr;
    size_t stage_bytes = 0;
    HostPipe pipe;
};

namespace {

// Keeps the caller's current device unchanged across a call made on h->device.
struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) return;
        ok = (prev == dev) || (cudaSetDevice(dev) == cudaSuccess);
    }
    ~DeviceGuard()
    {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

// Encode a 2-D row-major tensor map: `inner` contiguous elements per row, `outer` rows
// `pitch_bytes` apart, box = box_inner x box_outer, 128-byte swizzle (or none), zero fill
// outside.  With a cache (a handle's), identical requests reuse the earlier encoding.
bool get_tmap(std::vector<TmapEntry>* cache, const void* ptr, uint64_t inner, uint64_t outer, uint64_t pitch_bytes,
              uint32_t box_inner, uint32_t box_outer, int32_t dtype, CUtensorMap* out,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B)
{
    const TmapKey key{ptr, inner, outer, pitch_bytes, box_inner, box_outer, dtype, static_cast<int32_t>(swizzle)};
    if (cache)
        for (const TmapEntry& e : *cache)
            if (e.key == key) {
                *out = e.map;
                return true;
            }
    if (!load_encode_fn()) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {pitch_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    // 8-bit floats travel as bytes: TMA only moves them, the MMA interprets them.
    // kTmapBytes: raw bytes (side data).
    const CUtensorMapDataType dt = dtype == GEMM_DTYPE_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : dtype == GEMM_DTYPE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                             : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if (g_encode(out, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    if (cache) {
        if (static_cast<int>(cache->size()) >= kTmapCacheMax) cache->clear();
        cache->push_back({key, *out});
    }
    return true;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool is_f8(gemm_dtype_t t) { return t == GEMM_DTYPE_E4M3 || t == GEMM_DTYPE_E5M2; }
int elem_bytes(gemm_dtype_t t) { return is_f8(t) ? 1 : 2; }

// Kernel families beyond the dense one: block-scaled 8-bit operands, 2:4-sparse A (each with
// the one-CTA 128 x 256 tile and the CTA pair).
enum Family { kDense = 0, kBlockScaled = 1, kSparse24 = 2 };

// `out` is the type of C: equal to `in` for 16-bit operands, F16 or BF16 for 8-bit ones.
KernelChoice kernel_choice(int config, gemm_dtype_t in, gemm_dtype_t out, gemm_layout_t layout, int family = kDense)
{
    const bool nn = layout == GEMM_LAYOUT_NN, out_bf16 = out == GEMM_DTYPE_BF16;
    if (family == kBlockScaled) return dtg::choice_mx(config, in == GEMM_DTYPE_E5M2, out_bf16, nn);
    if (family == kSparse24) return dtg::choice_sparse(config, in == GEMM_DTYPE_BF16, nn);
    switch (in) {
    case GEMM_DTYPE_BF16: return dtg::choice_bf16(config, nn);
    case GEMM_DTYPE_E4M3: return dtg::choice_e4m3(config, out_bf16, nn);
    case GEMM_DTYPE_E5M2: return dtg::choice_e5m2(config, out_bf16, nn);
    default: return dtg::choice_f16(config, nn);
    }
}

int slot_of(int config, gemm_dtype_t in, gemm_dtype_t out, gemm_layout_t layout, int family = kDense)
{
    const int c = config == GEMM_CONFIG_128x64    ? 3
                  : config == GEMM_CONFIG_256x256 ? 2
                  : config == GEMM_CONFIG_128x128 ? 1 : 0;
    const int f8 = 2 * (in - GEMM_DTYPE_E4M3) + (out == GEMM_DTYPE_BF16 ? 1 : 0);  // 0..3
    const int types = family == kSparse24 ? 10 + in : (is_f8(in) ? (family == kBlockScaled ? 6 : 2) + f8 : in);
    return (c * 12 + types) * 2 + (layout == GEMM_LAYOUT_NN ? 1 : 0);
}

// Opt the kernel into its shared memory and, for pair kernels, ask how many clusters can
// be resident at once (the persistent grid never exceeds that).  Once per device and slot.
gemm_status_t ensure_kernel_ready(DeviceState& dev, const KernelChoice& kc, int slot)
{
    std::lock_guard<std::mutex> lock(dev.mu);
    if (!dev.attrs_set[slot]) {
        if (cudaFuncSetAttribute(kc.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kc.smem) != cudaSuccess)
            return GEMM_ERR_CUDA;
        if (kc.cluster > 1) {
            cudaLaunchConfig_t cfg;
            std::memset(&cfg, 0, sizeof(cfg));
            cfg.gridDim = dim3(static_cast<unsigned>(kc.cluster * (dev.num_sms / kc.cluster)), 1, 1);
            cfg.blockDim = dim3(static_cast<unsigned>(kc.threads), 1, 1);
            cfg.dynamicSmemBytes = static_cast<size_t>(kc.smem);
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = static_cast<unsigned>(kc.cluster);
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = 1;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kc.fn, &cfg) != cudaSuccess || n <= 0) return GEMM_ERR_CUDA;
            dev.max_clusters[slot] = n;
        }
        dev.attrs_set[slot] = true;
    }
    return GEMM_OK;
}

int pick_config(const LaunchOptions& o, const DeviceState& dev, int64_t M, int64_t N, int64_t K)
{
    if (o.config == GEMM_CONFIG_128x256 || o.config == GEMM_CONFIG_128x128 || o.config == GEMM_CONFIG_256x256 ||
        o.config == GEMM_CONFIG_128x64)
        return static_cast<int>(o.config);
    // AUTO: the 256 x 256 CTA-pair tile when there is at least one pair tile per pair of
    // SMs (it halves each SM's shared-memory traffic for B); otherwise the 128 x 256 tile
    // unless that leaves most SMs idle, then 128 x 128.  Below half a wave of those, a short
    // K loop runs on 128 x 64 tiles (more SMs taking in operands: 1000^3, 64 tiles of
    // 128 x 128 or 128 of 128 x 64, cold L2: 14.0 against 12.7 us), a long one (64 K blocks or
    // more) stays on 128 x 128 tiles whose K blocks fill_plan splits between CTAs (1000 x 1000
    // x 8192: 43.7 us on 128 whole 128 x 64 tiles, 34.4 us split over 152 CTAs).
    const int64_t pair_tiles = cdiv(M, 256) * cdiv(N, 256);
    if (pair_tiles >= dev.num_sms / 2) return GEMM_CONFIG_256x256;
    const int64_t tiles256 = cdiv(M, 128) * cdiv(N, 256);
    if (tiles256 >= dev.num_sms / 2) return GEMM_CONFIG_128x256;
    const int64_t tiles128 = cdiv(M, 128) * cdiv(N, 128);
    if (tiles128 >= dev.num_sms / 2 || cdiv(K, 64) >= 64) return GEMM_CONFIG_128x128;
    return GEMM_CONFIG_128x64;
}

// Workspace a stream-K plan with `units` work units needs (see the kernel's slot layout).
size_t sk_partial_floats(int64_t units, const KernelChoice& kc)
{
    return static_cast<size_t>(2 * units) * static_cast<size_t>(kc.cluster) * dtg::kBM * static_cast<size_t>(kc.bn);
}

int64_t sk_counter_count(int64_t sk_tiles, const KernelChoice& kc) { return sk_tiles * kc.cluster; }

// `ws` == nullptr: no workspace, every tile is done whole (data-parallel).
void fill_plan(const LaunchOptions& o, const DeviceState& dev, int max_clusters, const Workspace* ws, int64_t M,
               int64_t N, int64_t K, const KernelChoice& kc, int family, gemm_plan_t* plan)
{
    std::memset(plan, 0, sizeof(*plan));
    plan->config = kc.config;
    plan->bm = kc.bm;
    plan->bn = kc.bn;
    plan->bk = kc.stage_k;
    plan->stages = kc.stages;
    plan->cluster = kc.cluster;
    plan->tiles_m = cdiv(M, kc.bm);
    plan->tiles_n = cdiv(N, kc.bn);
    plan->k_blocks = cdiv(K, kc.stage_k);
    // Raster group: tile rows walked together.  Automatic: the tile rows whose A holds about
    // kGroupPanelBytes (the group's A stays in L2 while its B columns stream), at most
    // kMaxAutoGroup and at most as many rows as the grid has tile columns.  Measured at 8192^3
    // with every second item's K loop walked backwards: bf16 (4 MiB of A per tile row) runs
    // fastest with 12 rows (1926 TF/s burst, 1657 sustained, against 1917 / 1645 at 8, 1918 /
    // 1651 at 16, 1861 / 1600 at 4); a 2:4-compressed A (2 MiB) with 12-16 (2300 against 2289
    // at 8); E4M3 (2 MiB, forward K loops) with 16 (3555 against 3506 at 8, 3538 at 12);
    // 16384 x 1024 x 8192 fp16, 4 tile columns, with 4 (0.40 GB of DRAM per launch against
    // 0.57 at 8 and 0.66 at 1).
    const int64_t a_row_bytes = K * 128 / kc.stage_k * kc.a_stage_k / kc.stage_k;  // per matrix row (2:4: compressed)
    const int64_t panel = kc.bm * (a_row_bytes > 0 ? a_row_bytes : 1);
    const int64_t group = std::min<int64_t>(std::max<int64_t>(1, (kGroupPanelBytes + panel / 2) / panel), kMaxAutoGroup);
    plan->raster_group = o.raster_group > 0 ? o.raster_group : std::min<int64_t>(group, plan->tiles_n);
    // Block-scaled kernels walk every item's K blocks forward: each scale box covers the four
    // K blocks from the one a slot starts at.
    plan->k_snake = (o.k_snake && family != kBlockScaled) ? 1 : 0;
    const int64_t tiles = plan->tiles_m * plan->tiles_n;
    // Clusters (CTA pairs, or single CTAs) that can run at once, capped by the option.
    int64_t units = kc.cluster > 1 ? (max_clusters > 0 ? max_clusters : dev.num_sms / kc.cluster)
                                   : (dev.num_sms > 0 ? dev.num_sms : 1);
    if (o.max_ctas > 0) {
        const int64_t cap = o.max_ctas / kc.cluster;
        units = cap < 1 ? 1 : (cap < units ? cap : units);
    }
    if (units < 1) units = 1;
    plan->dp_tiles = tiles;
    // Stream-K when whole tiles would leave the last wave part-empty: every unit does
    // (full waves - 1) whole tiles, then an equal share of the K blocks of the rest.  A
    // share shorter than sk_min_blocks would cost more in partial-sum traffic than it saves.
    // A problem under one wave (fewer tiles than units) is split only when every share still
    // holds split_min_blocks and every tile gets at least two shares: the merge through the
    // workspace is a few microseconds of dependent global-memory traffic, so only long K loops
    // spread over many more units gain from it (measured, cold L2, 1000 x 1000 x K: 128 x 128
    // tiles at K = 1000 ran 13.6 us whole and 17.1 us as two 8-block shares per tile; at
    // K = 4096, 26.7 us whole and 23.8 us as two 32-block shares; 128 x 64 tiles, 128 of them,
    // were slower split over 152 CTAs at every K); fewer units then take shares of that
    // length.
    if (ws && o.stream_k && tiles % units != 0) {
        const int64_t dp = tiles >= units ? (tiles / units - 1) * units : 0;
        const int64_t sk_tiles = tiles - dp;
        const int64_t sk_blocks = sk_tiles * plan->k_blocks;
        int64_t sk_units = units;
        int64_t min_share = o.sk_min_blocks;
        if (tiles < units) {
            min_share = o.split_min_blocks > 0 ? o.split_min_blocks : sk_blocks + 1;  // 0: never split
            if (sk_blocks / units < min_share) sk_units = sk_blocks / min_share;
            if (sk_units < 2 * tiles) {  // fewer than two shares a tile: whole tiles
                sk_units = units;
                min_share = sk_blocks + 1;
            }
        }
        const int64_t base = sk_blocks / sk_units;
        if (base >= min_share && sk_partial_floats(sk_units, kc) <= ws->partial_floats &&
            sk_counter_count(sk_tiles, kc) <= ws->counter_count) {
            units = sk_units;
            plan->dp_tiles = dp;
            plan->sk_base = base;
            plan->sk_extra = sk_blocks % sk_units;
        }
    }
    if (plan->dp_tiles == tiles && tiles < units) units = tiles;  // whole tiles only: no idle units
    plan->grid = units * kc.cluster;
    plan->threads = kc.threads;
    plan->smem_bytes = kc.smem;
}

// c_col_major: C is stored N x M (C[m, n] at C + n * ldc + m), so ldc must cover M.
// out_dtype < 0: gemm_run's rule, 16-bit operands and C of the same type.  Otherwise any
// operand type, C of type out_dtype (16-bit), equal to dtype for 16-bit operands.
// sparse_a: A is the compressed 2:4 matrix, K / 2 columns (K a multiple of 4).
gemm_status_t validate_args(const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K,
                            int64_t lda, int64_t ldb, int64_t ldc, gemm_layout_t layout, gemm_dtype_t dtype,
                            bool c_col_major = false, gemm_dtype_t out_dtype = -1, bool sparse_a = false)
{
    if (layout != GEMM_LAYOUT_NN && layout != GEMM_LAYOUT_TN) return GEMM_ERR_INVALID_ARG;
    if (out_dtype < 0) {
        if (dtype != GEMM_DTYPE_F16 && dtype != GEMM_DTYPE_BF16) return GEMM_ERR_INVALID_ARG;
    } else {
        if (dtype != GEMM_DTYPE_F16 && dtype != GEMM_DTYPE_BF16 && !is_f8(dtype)) return GEMM_ERR_INVALID_ARG;
        if (out_dtype != GEMM_DTYPE_F16 && out_dtype != GEMM_DTYPE_BF16) return GEMM_ERR_INVALID_ARG;
        if (!is_f8(dtype) && out_dtype != dtype) return GEMM_ERR_INVALID_ARG;
    }
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C || ldc < (c_col_major ? M : N)) return GEMM_ERR_INVALID_ARG;
    if (K > 0) {
        if (!A || !B) return GEMM_ERR_INVALID_ARG;
        if (lda < (sparse_a ? K / 2 : K)) return GEMM_ERR_INVALID_ARG;
        if (ldb < (layout == GEMM_LAYOUT_NN ? N : K)) return GEMM_ERR_INVALID_ARG;
    }
    const int64_t lim = (int64_t(1) << 31) - 1;
    if (M > lim || N > lim || K > lim) return GEMM_ERR_UNSUPPORTED;
    if (sparse_a && K % 4 != 0) return GEMM_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(C) & 15u) != 0 || (ldc & 7) != 0) return GEMM_ERR_UNSUPPORTED;
    if (K > 0) {
        if ((reinterpret_cast<uintptr_t>(A) & 15u) != 0 || (reinterpret_cast<uintptr_t>(B) & 15u) != 0)
            return GEMM_ERR_UNSUPPORTED;
        // Row pitches of A and B are TMA strides: multiples of 16 bytes.
        const int64_t mask = 16 / elem_bytes(dtype) - 1;
        if ((lda & mask) != 0 || (ldb & mask) != 0) return GEMM_ERR_UNSUPPORTED;
    }
    return GEMM_OK;
}

gemm_status_t validate(gemm_handle_t h, const void* A, const void* B, const void* C, int64_t M, int64_t N,
                       int64_t K, int64_t lda, int64_t ldb, int64_t ldc, gemm_layout_t layout,
                       gemm_dtype_t dtype)
{
    if (!h) return GEMM_ERR_INVALID_ARG;
    return validate_args(A, B, C, M, N, K, lda, ldb, ldc, layout, dtype);
}

// The configuration launch_gemm runs for a problem with operands of kind `family`.
int choose_config(const LaunchOptions& o, const DeviceState& dev, int64_t M, int64_t N, int64_t K,
                  gemm_dtype_t dtype, int family)
{
    // Sparse and block-scaled kernels: the CTA pair where the dense choice would take it (or
    // when asked), else the one-CTA 128 x 256 tile (measured with the side-data warp and
    // 128-byte side-data rows: block-scaled, the pair gains 6-9 % at 8192^3, 5-12 % at 6144^3,
    // ties at 4096^3; sparse: the pair 2236 TF/s at 8192^3).  The pair addresses the side data
    // by rows of kSideRowBytes with 32-bit TMA coordinates, which must fit.
    int config = pick_config(o, dev, M, N, K);
    if (family == kBlockScaled && config == GEMM_CONFIG_128x128) config = GEMM_CONFIG_128x256;
    // An N-major 8-bit B row is 128 elements wide: 8-bit operands take 128 x 128 for 128 x 64.
    if (config == GEMM_CONFIG_128x64 && is_f8(dtype)) config = GEMM_CONFIG_128x128;
    if (family != kDense) {
        const int64_t lim = int64_t(1) << 31;
        const bool rows_fit =
            family == kSparse24
                ? cdiv(M, dtg::kBM) * cdiv(K, 64) * (dtg::kMetaChunkBytes / dtg::kSideRowBytes) < lim
                : (M > N ? cdiv(M, dtg::kBM) : cdiv(N, dtg::kBM)) * cdiv(K, 128) * (dtg::kSfChunkBytes / dtg::kSideRowBytes) <
                      lim;
        config = (config == GEMM_CONFIG_256x256 && rows_fit) ? config : GEMM_CONFIG_128x256;
    }
    return config;
}

// Enqueue C = A·B (arguments already validated, M, N > 0) on the current device.
// `ws` == nullptr restricts the schedule to whole tiles (no stream-K workspace).
gemm_status_t launch_gemm(const LaunchOptions& o, DeviceState& dev, const Workspace* ws,
                          std::vector<TmapEntry>* cache, int32_t* err,
                          const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                          int64_t ldb, int64_t ldc, gemm_layout_t layout, gemm_dtype_t dtype, cudaStream_t stream,
                          const Epilogue& ep = Epilogue())
{
    const gemm_dtype_t out = ep.out < 0 ? dtype : ep.out;
    if (K == 0) {
        int blocks = static_cast<int>(cdiv(M * N, 256));
        const int cap = dev.num_sms * 8;
        if (blocks > cap) blocks = cap;
        uint16_t* c16 = static_cast<uint16_t*>(C);
        if (out == GEMM_DTYPE_BF16)
            dtg::scale_c_kernel<true><<<blocks, 256, 0, stream>>>(c16, M, N, ldc, ep.col_major, ep.beta);
        else
            dtg::scale_c_kernel<false><<<blocks, 256, 0, stream>>>(c16, M, N, ldc, ep.col_major, ep.beta);
        return cudaPeekAtLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
    }

    const int family = ep.sfa ? kBlockScaled : (ep.meta ? kSparse24 : kDense);
    const int config = choose_config(o, dev, M, N, K, dtype, family);
    const KernelChoice kc = kernel_choice(config, dtype, out, layout, family);
    const int slot = slot_of(config, dtype, out, layout, family);
    const gemm_status_t ready = ensure_kernel_ready(dev, kc, slot);
    if (ready != GEMM_OK) return ready;
    gemm_plan_t plan;
    fill_plan(o, dev, dev.max_clusters[slot], ws, M, N, K, kc, family, &plan);

    CUtensorMap tA, tB, tC;
    const bool nn = layout == GEMM_LAYOUT_NN;
    const uint64_t eb = static_cast<uint64_t>(elem_bytes(dtype));
    const uint32_t sk = static_cast<uint32_t>(kc.stage_k);
    // A: K elements per row, or K / 2 for the compressed 2:4 matrix (64-byte stage rows,
    // 64-byte swizzle).
    const bool a_sw64 = static_cast<uint64_t>(kc.a_stage_k) * eb == 64;
    if (!get_tmap(cache, A, family == kSparse24 ? K / 2 : K, M, lda * eb, static_cast<uint32_t>(kc.a_stage_k), dtg::kBM,
                  dtype, &tA, a_sw64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B))
        return GEMM_ERR_CUDA;
    if (nn) {
        if (!get_tmap(cache, B, N, K, ldb * eb, static_cast<uint32_t>(kc.n_block), sk, dtype, &tB))
            return GEMM_ERR_CUDA;
    } else {
        if (!get_tmap(cache, B, K, N, ldb * eb, sk, static_cast<uint32_t>(kc.b_box), dtype, &tB))
            return GEMM_ERR_CUDA;
    }
    if (ep.col_major) {
        // C stored N x M: boxes of 32 (M, contiguous) x 64 (N), unswizzled.
        if (!get_tmap(cache, C, M, N, ldc * 2, 32, dtg::kEpiCols, out, &tC, CU_TENSOR_MAP_SWIZZLE_NONE))
            return GEMM_ERR_CUDA;
    } else if (!get_tmap(cache, C, N, M, ldc * 2, dtg::kEpiCols, 32, out, &tC)) {
        return GEMM_ERR_CUDA;
    }

    KernelParams kp;
    kp.M = static_cast<int32_t>(M);
    kp.N = static_cast<int32_t>(N);
    kp.K = static_cast<int32_t>(K);
    kp.tiles_m = static_cast<int32_t>(plan.tiles_m);
    kp.tiles_n = static_cast<int32_t>(plan.tiles_n);
    kp.num_kb = static_cast<int32_t>(plan.k_blocks);
    kp.num_tiles = static_cast<int32_t>(plan.tiles_m * plan.tiles_n);
    kp.group_m = static_cast<int32_t>(plan.raster_group);
    kp.fault_inject = static_cast<int32_t>(o.fault_inject);
    kp.k_snake = static_cast<int32_t>(plan.k_snake);
    kp.timeout_ns = static_cast<uint64_t>(o.timeout_ns);
    kp.err = err;
    kp.C = C;
    kp.ldc = ldc;
    kp.dp_tiles = static_cast<int32_t>(plan.dp_tiles);
    kp.sk_base = plan.sk_base;
    kp.sk_extra = plan.sk_extra;
    kp.ws = ws ? ws->partials : nullptr;
    kp.counters = ws ? ws->counters : nullptr;
    kp.alpha = ep.alpha;
    kp.beta = ep.beta;
    kp.c_col_major = ep.col_major;
    kp.sfa = static_cast<const uint8_t*>(ep.sfa);
    kp.sfb = static_cast<const uint8_t*>(ep.sfb);
    kp.sfb_blocks = static_cast<int32_t>(cdiv(N, dtg::kSfChunkRows));
    kp.meta = static_cast<const uint8_t*>(ep.meta);

    // Side data of a CTA-pair kernel as rows of kSideRowBytes (128): the metadata chunks (a
    // box of one chunk, 32 rows, per stage and CTA), or the A and B scale chunks (boxes of 4
    // rows).  Wide rows keep each box a few long transfers instead of many 16-byte ones.
    CUtensorMap tS = tA, tS2 = tA;
    if (family == kSparse24 && kc.cluster >= 2) {
        constexpr uint32_t kRb = dtg::kSideRowBytes;
        const uint64_t rows = static_cast<uint64_t>(cdiv(M, dtg::kBM) * cdiv(K, 64)) * (dtg::kMetaChunkBytes / kRb);
        if (!get_tmap(cache, ep.meta, kRb, rows, kRb, kRb, dtg::kMetaChunkBytes / kRb, kTmapBytes, &tS,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
            return GEMM_ERR_CUDA;
    }
    // Block scales (every block-scaled kernel): boxes of kScGroup consecutive chunks of one
    // row block, i.e. the scales of kScGroup ring stages (past the end of a row block the box
    // reads the next block's chunks, or zeros past the buffer; the kernel uses neither).
    if (family == kBlockScaled) {
        constexpr uint32_t kRb = dtg::kSideRowBytes;
        constexpr uint32_t kRows = dtg::kSfChunkBytes / kRb;
        const uint64_t rows_a = static_cast<uint64_t>(cdiv(M, dtg::kSfChunkRows) * cdiv(K, 128)) * kRows;
        const uint64_t rows_b = static_cast<uint64_t>(cdiv(N, dtg::kSfChunkRows) * cdiv(K, 128)) * kRows;
        if (rows_a >= (uint64_t(1) << 31) || rows_b >= (uint64_t(1) << 31)) return GEMM_ERR_UNSUPPORTED;
        if (!get_tmap(cache, ep.sfa, kRb, rows_a, kRb, kRb, kRows * dtg::kScGroup, kTmapBytes, &tS,
                      CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !get_tmap(cache, ep.sfb, kRb, rows_b, kRb, kRb, kRows * dtg::kScGroup, kTmapBytes, &tS2,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
            return GEMM_ERR_CUDA;
    }
    void* args[] = {&tA, &tB, &tC, &tS, &tS2, &kp};
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(plan.grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(kc.threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(kc.smem);
    cfg.stream = stream;
    // Programmatic dependent launch: the grid may be scheduled while the stream's previous
    // kernel finishes; the kernel runs its prologue, then waits (griddepcontrol.wait) for that
    // kernel's completion before it touches global memory.
    cudaLaunchAttribute attrs[2];
    unsigned n_attrs = 0;
    attrs[n_attrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n_attrs].val.programmaticStreamSerializationAllowed = 1;
    ++n_attrs;
    if (kc.cluster > 1) {
        attrs[n_attrs].id = cudaLaunchAttributeClusterDimension;
        attrs[n_attrs].val.clusterDim.x = static_cast<unsigned>(kc.cluster);
        attrs[n_attrs].val.clusterDim.y = 1;
        attrs[n_attrs].val.clusterDim.z = 1;
        ++n_attrs;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = n_attrs;
    if (cudaLaunchKernelExC(&cfg, kc.fn, args) != cudaSuccess) return GEMM_ERR_CUDA;
    return GEMM_OK;
}

gemm_status_t read_error_word(gemm_handle_t h, cudaStream_t stream)
{
    int32_t info[4] = {0, 0, 0, 0};
    if (cudaMemcpyAsync(info, h->d_err, sizeof(info), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GEMM_ERR_CUDA;
    if (info[0] != 0) {
        std::memcpy(h->last_info, info, sizeof(info));
        if (cudaMemsetAsync(h->d_err, 0, sizeof(info), stream) != cudaSuccess) return GEMM_ERR_CUDA;
        // An abandoned launch may have left stream-K arrival counters part-way.
        if (h->ws.counters &&
            cudaMemsetAsync(h->ws.counters, 0, static_cast<size_t>(h->ws.counter_count) * sizeof(int32_t), stream) !=
                cudaSuccess)
            return GEMM_ERR_CUDA;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return GEMM_ERR_CUDA;
        return GEMM_ERR_TIMEOUT;
    }
    return GEMM_OK;
}

// Compute capability and SM count of `device`; ARCH unless it is sm_103.
gemm_status_t query_device(int device, int* sms)
{
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (major != 10 || minor != 3) return GEMM_ERR_ARCH;
    return GEMM_OK;
}

// Block scales, row-major (src[r * ld + j]: the exponent of K block j of row r, rows x
// kblocks) -> the chunked layout the block-scaled kernels load (dtg::kSfChunkBytes).  Rows and K
// blocks past the end are filled with 127 (a scale of 1: padded K elements are zero and stay
// zero).  Grid-stride over the `total` destination bytes.
__global__ void pack_scales_kernel(const uint8_t* src, int64_t rows, int64_t kblocks, int64_t ld, uint8_t* dst,
                                   int64_t total)
{
    const int64_t groups = (kblocks + 3) / 4;
    for (int64_t o = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; o < total;
         o += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t chunk = o / dtg::kSfChunkBytes;
        const int within = static_cast<int>(o - chunk * dtg::kSfChunkBytes);
        const int64_t rb = chunk / groups, g = chunk - rb * groups;
        const int64_t r = rb * dtg::kSfChunkRows + ((within >> 2) & 3) * 32 + (within >> 4);
        const int64_t j = g * 4 + (within & 3);
        dst[o] = (r < rows && j < kblocks) ? src[r * ld + j] : static_cast<uint8_t>(127);
    }
}

// Metadata word of row r for groups [8 j, 8 j + 8) (K [32 j, 32 j + 32)) and the kept values:
// per group of four the first two non-zero codes (a code is zero when all bits but the sign
// are 0) are kept, the lowest free positions complete the pair, the pair is put in ascending
// order; Ac gets the two values.  Groups past K and rows past M get the pattern (0, 1) and no
// values.  Returns the number of groups with more than two non-zeros.
__device__ int32_t sparse24_word(const uint16_t* A, int64_t M, int64_t K, int64_t lda, uint16_t* Ac, int64_t ldac,
                                 int64_t r, int64_t j, uint32_t* word)
{
    const int64_t groups = K / 4;
    uint32_t w = 0;
    int32_t nbad = 0;
    for (int q = 0; q < 8; ++q) {
        const int64_t g = 8 * j + q;
        uint32_t nib = 0x4u;  // positions (0, 1)
        if (r < M && g < groups) {
            const uint16_t* a = A + r * lda + 4 * g;
            int p0 = -1, p1 = -1, nonzero = 0;
            for (int i = 0; i < 4; ++i)
                if ((a[i] & 0x7fffu) != 0u) {
                    ++nonzero;
                    if (p0 < 0)
                        p0 = i;
                    else if (p1 < 0)
                        p1 = i;
                }
            if (nonzero > 2) ++nbad;
            for (int i = 0; p1 < 0 && i < 4; ++i)
                if (p0 < 0)
                    p0 = i;
                else if (i != p0)
                    p1 = i;
            if (p0 > p1) {
                const int tmp = p0;
                p0 = p1;
                p1 = tmp;
            }
            Ac[r * ldac + 2 * g] = a[p0];
            Ac[r * ldac + 2 * g + 1] = a[p1];
            nib = static_cast<uint32_t>(p0 | (p1 << 2));
        }
        w |= nib << (4 * q);
    }
    *word = w;
    return nbad;
}

// 2:4 compression of a dense 16-bit A (M x K, K % 4 == 0) into Ac and the metadata chunks
// (dtg::kMetaChunkBytes).  One thread per (row pair, ring stage of 64 K): rows r = 16 b + i
// and r + 8 (i < 8) share TMEM words, as the sparse MMA reads them: in the half of MMA h,
// lane r holds groups 0-3 of the MMA's 32 K for row r (low 16 bits) and for row r + 8 (high
// 16 bits), lane r + 8 holds groups 4-7 of both rows the same way; three padding words
// follow each word.  Groups with more than two non-zeros are counted into *bad (if not null).
__global__ void sparse24_compress_kernel(const uint16_t* A, int64_t M, int64_t K, int64_t lda, uint16_t* Ac,
                                         int64_t ldac, uint8_t* meta, int32_t* bad, int64_t rows_pad, int64_t stages)
{
    const int64_t pairs = rows_pad / 2;
    const int64_t total = pairs * stages;
    for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < total;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t pi = t % pairs, s = t / pairs;
        const int64_t r = 16 * (pi / 8) + pi % 8, r2 = r + 8;
        int32_t nbad = 0;
        uint8_t* chunk = meta + ((r / dtg::kBM) * stages + s) * dtg::kMetaChunkBytes;
        for (int h = 0; h < 2; ++h) {
            uint32_t w1, w2;
            nbad += sparse24_word(A, M, K, lda, Ac, ldac, r, 2 * s + h, &w1);
            nbad += sparse24_word(A, M, K, lda, Ac, ldac, r2, 2 * s + h, &w2);
            uint8_t* half = chunk + h * dtg::kMetaHalfBytes;
            *reinterpret_cast<uint4*>(half + (r % dtg::kBM) * 16) =
                make_uint4((w1 & 0xFFFFu) | (w2 << 16), 0x44444444u, 0x44444444u, 0x44444444u);
            *reinterpret_cast<uint4*>(half + (r2 % dtg::kBM) * 16) =
                make_uint4((w1 >> 16) | (w2 & 0xFFFF0000u), 0x44444444u, 0x44444444u, 0x44444444u);
        }
        if (nbad && bad) atomicAdd(bad, nbad);
    }
}

// Boundaries of `wanted` (at most) equal chunks of an extent, each a multiple of 256 long
// (whole pair tiles) and at least `min_size` long, except the last: bounds[0] = 0,
// bounds[n] = extent; returns n.
int host_chunks(int64_t extent, int64_t wanted, int64_t min_size, int64_t* bounds)
{
    const int64_t size = std::max<int64_t>(min_size, (cdiv(extent, wanted) + 255) / 256 * 256);
    const int n = static_cast<int>(cdiv(extent, size));
    for (int i = 0; i <= n; ++i) bounds[i] = std::min<int64_t>(static_cast<int64_t>(i) * size, extent);
    return n;
}

}  // namespace

extern "C" {

gemm_status_t gemm_create(gemm_handle_t* out, int device)
{
    if (!out) return GEMM_ERR_INVALID_ARG;
    *out = nullptr;
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (device < 0 || device >= count) return GEMM_ERR_INVALID_ARG;
    int sms = 0;
    const gemm_status_t q = query_device(device, &sms);
    if (q != GEMM_OK) return q;
    DeviceGuard g(device);
    if (!g.ok) return GEMM_ERR_CUDA;
    gemm_handle_s* h = new (std::nothrow) gemm_handle_s();
    if (!h) return GEMM_ERR_CUDA;
    h->device = device;
    h->dev.num_sms = sms;
    // Stream-K workspace, sized for the largest plan any configuration makes on this
    // device: 2 slots per work unit of 128 x 256 fp32 per CTA, and an arrival counter per
    // stream-K tile (at most two waves of tiles) and CTA.
    h->ws.partial_floats = static_cast<size_t>(2 * sms) * dtg::kBM * 256;
    h->ws.counter_count = 4 * static_cast<int64_t>(sms);
    if (cudaMalloc(&h->d_err, 4 * sizeof(int32_t)) != cudaSuccess ||
        cudaMemset(h->d_err, 0, 4 * sizeof(int32_t)) != cudaSuccess ||
        cudaMalloc(&h->ws.partials, h->ws.partial_floats * sizeof(float)) != cudaSuccess ||
        cudaMalloc(&h->ws.counters, static_cast<size_t>(h->ws.counter_count) * sizeof(int32_t)) != cudaSuccess ||
        cudaMemset(h->ws.counters, 0, static_cast<size_t>(h->ws.counter_count) * sizeof(int32_t)) != cudaSuccess) {
        if (h->d_err) cudaFree(h->d_err);
        if (h->ws.partials) cudaFree(h->ws.partials);
        if (h->ws.counters) cudaFree(h->ws.counters);
        delete h;
        return GEMM_ERR_CUDA;
    }
    *out = h;
    return GEMM_OK;
}

gemm_status_t gemm_destroy(gemm_handle_t h)
{
    if (!h) return GEMM_OK;
    gemm_status_t st = GEMM_OK;
    {
        DeviceGuard g(h->device);
        if (cudaDeviceSynchronize() != cudaSuccess) st = GEMM_ERR_CUDA;
        if (h->d_err && cudaFree(h->d_err) != cudaSuccess) st = GEMM_ERR_CUDA;
        if (h->d_stage && cudaFree(h->d_stage) != cudaSuccess) st = GEMM_ERR_CUDA;
        if (h->ws.partials && cudaFree(h->ws.partials) != cudaSuccess) st = GEMM_ERR_CUDA;
        if (h->ws.counters && cudaFree(h->ws.counters) != cudaSuccess) st = GEMM_ERR_CUDA;
        if (h->pipe.ready) {
            for (cudaStream_t q : {h->pipe.in, h->pipe.out}) cudaStreamDestroy(q);
            for (cudaEvent_t e : {h->pipe.start, h->pipe.done}) cudaEventDestroy(e);
            for (int i = 0; i < HostPipe::kMaxPieces; ++i) {
                cudaEventDestroy(h->pipe.arrived[i]);
                cudaEventDestroy(h->pipe.computed[i]);
            }
        }
    }
    delete h;
    return st;
}

gemm_status_t gemm_run(gemm_handle_t h, const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                       int64_t lda, int64_t ldb, int64_t ldc, gemm_layout_t layout, gemm_dtype_t dtype,
                       void* stream)
{
    const gemm_status_t v = validate(h, A, B, C, M, N, K, lda, ldb, ldc, layout, dtype);
    if (v != GEMM_OK || M == 0 || N == 0) return v;
    DeviceGuard g(h->device);
    if (!g.ok) return GEMM_ERR_CUDA;
    return launch_gemm(h->opts, h->dev, &h->ws, &h->tmaps, h->d_err, A, B, C, M, N, K, lda, ldb, ldc, layout, dtype,
                       static_cast<cudaStream_t>(stream));
}

// Checks of gemm_args_t shared by gemm_run_ex and gemm_run_mx; fills the epilogue.
static gemm_status_t validate_ex(const gemm_args_t& a, Epilogue* ep)
{
    if (a.c_col_major != 0 && a.c_col_major != 1) return GEMM_ERR_INVALID_ARG;
    if (a.out_dtype < 0) return GEMM_ERR_INVALID_ARG;
    // The three factors are multiplied in fp32 before the kernel scales the accumulator.
    const float alpha = a.alpha * a.scale_a * a.scale_b;
    if (!std::isfinite(a.alpha) || !std::isfinite(a.beta) || !std::isfinite(a.scale_a) ||
        !std::isfinite(a.scale_b) || !std::isfinite(alpha))
        return GEMM_ERR_INVALID_ARG;
    const gemm_status_t v = validate_args(a.A, a.B, a.C, a.M, a.N, a.K, a.lda, a.ldb, a.ldc, a.layout, a.dtype,
                                          a.c_col_major != 0, a.out_dtype);
    if (v != GEMM_OK) return v;
    ep->alpha = alpha;
    ep->beta = a.beta;
    ep->col_major = a.c_col_major;
    ep->out = a.out_dtype;
    return GEMM_OK;
}

gemm_status_t gemm_run_ex(gemm_handle_t h, const gemm_args_t* args, void* stream)
{
    if (!h || !args) return GEMM_ERR_INVALID_ARG;
    const gemm_args_t& a = *args;
    Epilogue ep;
    const gemm_status_t v = validate_ex(a, &ep);
    if (v != GEMM_OK || a.M == 0 || a.N == 0) return v;
    DeviceGuard g(h->device);
    if (!g.ok) return GEMM_ERR_CUDA;
    return launch_gemm(h->opts, h->dev, &h->ws, &h->tmaps, h->d_err, a.A, a.B, a.C, a.M, a.N, a.K, a.lda, a.ldb,
                       a.ldc, a.layout, a.dtype, static_cast<cudaStream_t>(stream), ep);
}

int64_t gemm_mx_scale_bytes(int64_t rows, int64_t K)
{
    if (rows <= 0 || K <= 0) return 0;
    return cdiv(rows, dtg::kSfChunkRows) * cdiv(K, 128) * dtg::kSfChunkBytes;
}

gemm_status_t gemm_run_mx(gemm_handle_t h, const gemm_args_t* args, const void* sfa, const void* sfb, void* stream)
{
    if (!h || !args) return GEMM_ERR_INVALID_ARG;
    const gemm_args_t& a = *args;
    if (!is_f8(a.dtype)) return GEMM_ERR_INVALID_ARG;
    Epilogue ep;
    const gemm_status_t v = validate_ex(a, &ep);
    if (v != GEMM_OK || a.M == 0 || a.N == 0) return v;
    if (a.K > 0) {
        if (!sfa || !sfb) return GEMM_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(sfa) & 15u) != 0 || (reinterpret_cast<uintptr_t>(sfb) & 15u) != 0)
            return GEMM_ERR_UNSUPPORTED;
        ep.sfa = sfa;
        ep.sfb = sfb;
    }
    DeviceGuard g(h->device);
    if (!g.ok) return GEMM_ERR_CUDA;
    return launch_gemm(h->opts, h->dev, &h->ws, &h->tmaps, h->d_err, a.A, a.B, a.C, a.M, a.N, a.K, a.lda, a.ldb,
                       a.ldc, a.layout, a.dtype, static_cast<cudaStream_t>(stream), ep);
}

int64_t gemm_sp_meta_bytes(int64_t M, int64_t K)
{
    if (M <= 0 || K <= 0) return 0;
    return cdiv(M, dtg::kBM) * cdiv(K, 64) * dtg::kMetaChunkBytes;
}

gemm_status_t gemm_sp_compress(gemm_handle_t h, const void* A, int64_t M, int64_t K, int64_t lda, gemm_dtype_t dtype,
                               void* Ac, int64_t ldac, void* meta, int32_t* bad_groups, void* stream)
{
    if (!h || M < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (dtype != GEMM_DTYPE_F16 && dtype != GEMM_DTYPE_BF16) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || K == 0) return GEMM_OK;
    if (K % 4 != 0) return GEMM_ERR_UNSUPPORTED;
    if (!A || !Ac || !meta || lda < K || ldac < K / 2) return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(meta) & 15u) != 0) return GEMM_ERR_UNSUPPORTED;
    DeviceGuard g(h->device);
    if (!g.ok) return GEMM_ERR_CUDA;
    const int64_t rows_pad = cdiv(M, dtg::kBM) * dtg::kBM, stages = cdiv(K, 64);
    int blocks = static_cast<int>(cdiv(rows_pad / 2 * stages, 256));
    const int cap = h->dev.num_sms * 8;
    if (blocks > cap) blocks = cap;
    sparse24_compress_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(A), M, K, lda, static_cast<uint16_t*>(Ac), ldac, static_cast<uint8_t*>(meta),
        bad_groups, rows_pad, stages);
    return cudaPeekAtLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

gemm_status_t gemm_run_sp(gemm_handle_t h, const gemm_args_t* args, const void* meta, void* stream)
{
    if (!h || !args) return GEMM_ERR_INVALID_ARG;
    const gemm_args_t& a = *args;
    if (a.dtype != GEMM_DTYPE_F16 && a.dtype != GEMM_DTYPE_BF16) return GEMM_ERR_INVALID_ARG;
    if (a.c_col_major != 0 && a.c_col_major != 1) return GEMM_ERR_INVALID_ARG;
    if (a.out_dtype != a.dtype) return GEMM_ERR_INVALID_ARG;
    const float alpha = a.alpha * a.scale_a * a.scale_b;
    if (!std::isfinite(a.alpha) || !std::isfinite(a.beta) || !std::isfinite(a.scale_a) ||
        !std::isfinite(a.scale_b) || !std::isfinite(alpha))
        return GEMM_ERR_INVALID_ARG;
    const gemm_status_t v = validate_args(a.A, a.B, a.C, a.M, a.N, a.K, a.lda, a.ldb, a.ldc, a.layout, a.dtype,
                                          a.c_col_major != 0, a.out_dtype, true);
    if (v != GEMM_OK || a.M == 0 || a.N == 0) return v;
    Epilogue ep;
    ep.alpha = alpha;
    ep.beta = a.beta;
    ep.col_major = a.c_col_major;
    ep.out = a.out_dtype;
    if (a.K > 0) {
        if (!meta) return GEMM_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(meta) & 15u) != 0) return GEMM_ERR_UNSUPPORTED;
        ep.meta = meta;
    }
    DeviceGuard g(h->device);
    if (!g.ok) return GEMM_ERR_CUDA;
    return launch_gemm(h->opts, h->dev, &h->ws, &h->tmaps, h->d_err, a.A, a.B, a.C, a.M, a.N, a.K, a.lda, a.ldb,
                       a.ldc, a.layout, a.dtype, static_cast<cudaStream_t>(stream), ep);
}

gemm_status_t gemm_mx_pack_scales(gemm_handle_t h, const void* src, int64_t rows, int64_t kblocks, int64_t ld,
                                  void* dst, void* stream)
{
    if (!h || rows < 0 || kblocks < 0) return GEMM_ERR_INVALID_ARG;
    if (rows == 0 || kblocks == 0) return GEMM_OK;
    if (!src || !dst || ld < kblocks) return GEMM_ERR_INVALID_ARG;
    const int64_t total = cdiv(rows, dtg::kSfChunkRows) * cdiv(kblocks, 4) * dtg::kSfChunkBytes;
    DeviceGuard g(h->device);
    if (!g.ok) return GEMM_ERR_CUDA;
    int blocks = static_cast<int>(cdiv(total, 256));
    const int cap = h->dev.num_sms * 8;
    if (blocks > cap) blocks = cap;
    pack_scales_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(src), rows, kblocks, ld, static_cast<uint8_t*>(dst), total);
    return cudaPeekAtLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

gemm_status_t gemm_run_host(gemm_handle_t h, const void* A, const void* B, void* C, int64_t M, int64_t N,
                            int64_t K, int64_t lda, int64_t ldb, int64_t ldc, gemm_layout_t layout,
                            gemm_dtype_t dtype, void* stream)
{
    const gemm_status_t v = validate(h, A, B, C, M, N, K, lda, ldb, ldc, layout, dtype);
    if (v != GEMM_OK || M == 0 || N == 0) return v;
    DeviceGuard g(h->device);
    if (!g.ok) return GEMM_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    HostPipe& hp = h->pipe;
    if (!hp.ready) {
        for (cudaStream_t* q : {&hp.in, &hp.out})
            if (cudaStreamCreateWithFlags(q, cudaStreamNonBlocking) != cudaSuccess) return GEMM_ERR_CUDA;
        for (cudaEvent_t* e : {&hp.start, &hp.done})
            if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return GEMM_ERR_CUDA;
        for (int i = 0; i < HostPipe::kMaxPieces; ++i)
            if (cudaEventCreateWithFlags(&hp.arrived[i], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&hp.computed[i], cudaEventDisableTiming) != cudaSuccess)
                return GEMM_ERR_CUDA;
        hp.ready = true;
    }
    // Device copies are packed: ld rounded up to 8 elements (16 bytes) keeps TMA alignment.
    auto r8 = [](int64_t x) { return (x + 7) & ~int64_t(7); };
    auto r256 = [](size_t x) { return (x + 255) & ~size_t(255); };
    const bool nn = layout == GEMM_LAYOUT_NN;
    const int64_t b_rows = nn ? K : N, b_cols = nn ? N : K;
    const int64_t dlda = r8(K > 0 ? K : 1), dldb = r8(b_cols > 0 ? b_cols : 1), dldc = r8(N);
    const size_t bytes_a = r256(static_cast<size_t>(M) * dlda * 2);
    const size_t bytes_b = r256(static_cast<size_t>(b_rows) * dldb * 2);
    const size_t bytes_c = r256(static_cast<size_t>(M) * dldc * 2);
    const size_t need = bytes_a + bytes_b + bytes_c;
    if (need > h->stage_bytes) {
        if (h->d_stage) {
            if (cudaStreamSynchronize(s) != cudaSuccess || cudaFree(h->d_stage) != cudaSuccess) return GEMM_ERR_CUDA;
            h->d_stage = nullptr;
            h->stage_bytes = 0;
        }
        if (cudaMalloc(&h->d_stage, need) != cudaSuccess) {
            h->d_stage = nullptr;
            return GEMM_ERR_CUDA;
        }
        h->stage_bytes = need;
    }
    char* dA = static_cast<char*>(h->d_stage);
    char* dB = dA + bytes_a;
    char* dC = dB + bytes_b;
    const char* hA = static_cast<const char*>(A);
    const char* hB = static_cast<const char*>(B);
    char* hC = static_cast<char*>(C);

    // Pipeline.  The host link, not the GPU, bounds this call, so the aim is to keep the
    // host-to-device copies running back to back and to copy C back while they run.  A is
    // split into row chunks and C's columns into column chunks (B's rows for TN, B's
    // columns for NN).  The inputs go over on one stream in the order B chunk 0, A chunk 0,
    // B chunk 1, A chunk 1, ... (the rest of the longer list last).  When a piece has
    // arrived, the GEMM of every block of C it completes is launched on `stream` (one
    // launch: the new A chunk against the B columns already in, or the new B chunk against
    // the A rows already in), and that block of C goes back on a third stream while later
    // pieces are still arriving.  Chunks are at least 1024 rows and 2048 columns, so each
    // launch still fills the GPU.  Measured on 8192^3 bf16 (a link of ~210 GB/s each way,
    // ~336 GB/s both ways at once; 1.30 ms for the inputs alone): 8 x 4 chunks 1.72 ms per
    // call, 4 x 2 1.76, 16 x 1 (512-row GEMMs that each stream all of B) 2.37.
    int64_t rb[HostPipe::kMaxRowChunks + 1], cb[HostPipe::kMaxColChunks + 1];
    const int nr = host_chunks(M, h->opts.host_row_chunks, 1024, rb);
    const int nc = host_chunks(N, h->opts.host_col_chunks, 2048, cb);
    struct Piece {
        bool a;  // a row chunk of A (else a column chunk of C's B)
        int idx;
    };
    Piece order[HostPipe::kMaxPieces];
    int np = 0;
    for (int k = 0; k < std::max(nr, nc); ++k) {
        if (k < nc) order[np++] = {false, k};
        if (k < nr) order[np++] = {true, k};
    }

    if (cudaEventRecord(hp.start, s) != cudaSuccess) return GEMM_ERR_CUDA;
    for (cudaStream_t q : {hp.in, hp.out})
        if (cudaStreamWaitEvent(q, hp.start, 0) != cudaSuccess) return GEMM_ERR_CUDA;
    int a_in = 0, b_in = 0, launches = 0;  // A / B chunks arrived so far (in order)
    for (int p = 0; p < np; ++p) {
        const Piece pc = order[p];
        if (K > 0) {
            cudaError_t e;
            if (pc.a) {
                const int64_t r0 = rb[pc.idx], rows = rb[pc.idx + 1] - r0;
                e = cudaMemcpy2DAsync(dA + r0 * dlda * 2, dlda * 2, hA + r0 * lda * 2, lda * 2, K * 2, rows,
                                      cudaMemcpyHostToDevice, hp.in);
            } else {
                const int64_t c0 = cb[pc.idx], cols = cb[pc.idx + 1] - c0;
                e = nn ? cudaMemcpy2DAsync(dB + c0 * 2, dldb * 2, hB + c0 * 2, ldb * 2, cols * 2, K,
                                           cudaMemcpyHostToDevice, hp.in)
                       : cudaMemcpy2DAsync(dB + c0 * dldb * 2, dldb * 2, hB + c0 * ldb * 2, ldb * 2, K * 2, cols,
                                           cudaMemcpyHostToDevice, hp.in);
            }
            if (e != cudaSuccess) return GEMM_ERR_CUDA;
        }
        if (cudaEventRecord(hp.arrived[p], hp.in) != cudaSuccess) return GEMM_ERR_CUDA;
        int64_t r0, r1, c0, c1;  // the block of C this piece completes
        if (pc.a) {
            ++a_in;
            r0 = rb[pc.idx], r1 = rb[pc.idx + 1], c0 = 0, c1 = cb[b_in];
        } else {
            ++b_in;
            r0 = 0, r1 = rb[a_in], c0 = cb[pc.idx], c1 = cb[pc.idx + 1];
        }
        if (r1 <= r0 || c1 <= c0) continue;
        if (cudaStreamWaitEvent(s, hp.arrived[p], 0) != cudaSuccess) return GEMM_ERR_CUDA;
        const char* bblk = nn ? dB + c0 * 2 : dB + c0 * dldb * 2;
        char* cblk = dC + (r0 * dldc + c0) * 2;
        const gemm_status_t st = launch_gemm(h->opts, h->dev, &h->ws, &h->tmaps, h->d_err, dA + r0 * dlda * 2, bblk,
                                             cblk, r1 - r0, c1 - c0, K, dlda, dldb, dldc, layout, dtype, s);
        if (st != GEMM_OK) return st;
        if (cudaEventRecord(hp.computed[launches], s) != cudaSuccess ||
            cudaStreamWaitEvent(hp.out, hp.computed[launches], 0) != cudaSuccess)
            return GEMM_ERR_CUDA;
        ++launches;
        if (cudaMemcpy2DAsync(hC + (r0 * ldc + c0) * 2, ldc * 2, cblk, dldc * 2, (c1 - c0) * 2, r1 - r0,
                              cudaMemcpyDeviceToHost, hp.out) != cudaSuccess)
            return GEMM_ERR_CUDA;
    }
    if (cudaEventRecord(hp.done, hp.out) != cudaSuccess || cudaStreamWaitEvent(s, hp.done, 0) != cudaSuccess)
        return GEMM_ERR_CUDA;
    return read_error_word(h, s);
}

gemm_status_t gemm_sync_status(gemm_handle_t h, void* stream)
{
    if (!h) return GEMM_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok) return GEMM_ERR_CUDA;
    return read_error_word(h, static_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_error_info(gemm_handle_t h, int32_t info[4])
{
    if (!h || !info) return GEMM_ERR_INVALID_ARG;
    std::memcpy(info, h->last_info, sizeof(h->last_info));
    return GEMM_OK;
}

gemm_status_t gemm_set_option(gemm_handle_t h, gemm_option_t opt, int64_t value)
{
    if (!h) return GEMM_ERR_INVALID_ARG;
    LaunchOptions& o = h->opts;
    switch (opt) {
    case GEMM_OPT_CONFIG:
        if (value != GEMM_CONFIG_AUTO && value != GEMM_CONFIG_128x256 && value != GEMM_CONFIG_128x128 &&
            value != GEMM_CONFIG_256x256 && value != GEMM_CONFIG_128x64)
            return GEMM_ERR_INVALID_ARG;
        o.config = value;
        return GEMM_OK;
    case GEMM_OPT_TIMEOUT_NS:
        if (value < 1000000) return GEMM_ERR_INVALID_ARG;
        o.timeout_ns = value;
        return GEMM_OK;
    case GEMM_OPT_MAX_CTAS:
        if (value < 0) return GEMM_ERR_INVALID_ARG;
        o.max_ctas = value;
        return GEMM_OK;
    case GEMM_OPT_RASTER_GROUP:
        if (value < 0 || value > (1 << 20)) return GEMM_ERR_INVALID_ARG;
        o.raster_group = value;
        return GEMM_OK;
    case GEMM_OPT_FAULT_INJECT:
        if (value != 0 && value != 1) return GEMM_ERR_INVALID_ARG;
        o.fault_inject = value;
        return GEMM_OK;
    case GEMM_OPT_STREAM_K:
        if (value != 0 && value != 1) return GEMM_ERR_INVALID_ARG;
        o.stream_k = value;
        return GEMM_OK;
    case GEMM_OPT_SK_MIN_BLOCKS:
        if (value < 1 || value > (1 << 20)) return GEMM_ERR_INVALID_ARG;
        o.sk_min_blocks = value;
        return GEMM_OK;
    case GEMM_OPT_SPLIT_MIN_BLOCKS:
        if (value < 0 || value > (1 << 20)) return GEMM_ERR_INVALID_ARG;
        o.split_min_blocks = value;
        return GEMM_OK;
    case GEMM_OPT_K_SNAKE:
        if (value != 0 && value != 1) return GEMM_ERR_INVALID_ARG;
        o.k_snake = value;
        return GEMM_OK;
    case GEMM_OPT_HOST_ROW_CHUNKS:
        if (value < 1 || value > HostPipe::kMaxRowChunks) return GEMM_ERR_INVALID_ARG;
        o.host_row_chunks = value;
        return GEMM_OK;
    case GEMM_OPT_HOST_COL_CHUNKS:
        if (value < 1 || value > HostPipe::kMaxColChunks) return GEMM_ERR_INVALID_ARG;
        o.host_col_chunks = value;
        return GEMM_OK;
    default:
        return GEMM_ERR_INVALID_ARG;
    }
}

gemm_status_t gemm_get_option(gemm_handle_t h, gemm_option_t opt, int64_t* value)
{
    if (!h || !value) return GEMM_ERR_INVALID_ARG;
    const LaunchOptions& o = h->opts;
    switch (opt) {
    case GEMM_OPT_CONFIG: *value = o.config; return GEMM_OK;
    case GEMM_OPT_TIMEOUT_NS: *value = o.timeout_ns; return GEMM_OK;
    case GEMM_OPT_MAX_CTAS: *value = o.max_ctas; return GEMM_OK;
    case GEMM_OPT_RASTER_GROUP: *value = o.raster_group; return GEMM_OK;
    case GEMM_OPT_FAULT_INJECT: *value = o.fault_inject; return GEMM_OK;
    case GEMM_OPT_STREAM_K: *value = o.stream_k; return GEMM_OK;
    case GEMM_OPT_SK_MIN_BLOCKS: *value = o.sk_min_blocks; return GEMM_OK;
    case GEMM_OPT_SPLIT_MIN_BLOCKS: *value = o.split_min_blocks; return GEMM_OK;
    case GEMM_OPT_K_SNAKE: *value = o.k_snake; return GEMM_OK;
    case GEMM_OPT_HOST_ROW_CHUNKS: *value = o.host_row_chunks; return GEMM_OK;
    case GEMM_OPT_HOST_COL_CHUNKS: *value = o.host_col_chunks; return GEMM_OK;
    default: return GEMM_ERR_INVALID_ARG;
    }
}

gemm_status_t gemm_query_plan_kind(gemm_handle_t h, int64_t M, int64_t N, int64_t K, gemm_layout_t layout,
                                   gemm_dtype_t dtype, gemm_kind_t kind, gemm_plan_t* plan)
{
    if (!h || !plan || M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (layout != GEMM_LAYOUT_NN && layout != GEMM_LAYOUT_TN) return GEMM_ERR_INVALID_ARG;
    const bool b16 = dtype == GEMM_DTYPE_F16 || dtype == GEMM_DTYPE_BF16;
    if (kind == GEMM_KIND_DENSE ? !(b16 || is_f8(dtype))
                                : kind == GEMM_KIND_BLOCK_SCALED ? !is_f8(dtype)
                                                                 : kind == GEMM_KIND_SPARSE24 ? !b16 : true)
        return GEMM_ERR_INVALID_ARG;
    // 8-bit operands: the plan of the bf16-output kernel (the fp16-output one is the same).
    const gemm_dtype_t out = is_f8(dtype) ? GEMM_DTYPE_BF16 : dtype;
    const int family = static_cast<int>(kind);  // gemm_kind_t and Family number the kinds alike
    DeviceGuard g(h->device);
    if (!g.ok) return GEMM_ERR_CUDA;
    const int config = choose_config(h->opts, h->dev, M, N, K, dtype, family);
    const KernelChoice kc = kernel_choice(config, dtype, out, layout, family);
    const int slot = slot_of(config, dtype, out, layout, family);
    const gemm_status_t ready = ensure_kernel_ready(h->dev, kc, slot);
    if (ready != GEMM_OK) return ready;
    fill_plan(h->opts, h->dev, h->dev.max_clusters[slot], &h->ws, M, N, K, kc, family, plan);
    return GEMM_OK;
}

gemm_status_t gemm_query_plan(gemm_handle_t h, int64_t M, int64_t N, int64_t K, gemm_layout_t layout,
                              gemm_dtype_t dtype, gemm_plan_t* plan)
{
    return gemm_query_plan_kind(h, M, N, K, layout, dtype, GEMM_KIND_DENSE, plan);
}

gemm_status_t gemm_check_args(const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K,
                              int64_t lda, int64_t ldb, int64_t ldc, gemm_layout_t layout, gemm_dtype_t dtype)
{
    return validate_args(A, B, C, M, N, K, lda, ldb, ldc, layout, dtype);
}

gemm_status_t gemm_tile_coord(int64_t tile, int64_t tiles_m, int64_t tiles_n, int64_t group_m, int64_t* tile_m,
                              int64_t* tile_n)
{
    if (!tile_m || !tile_n || tiles_m <= 0 || tiles_n <= 0 || group_m <= 0) return GEMM_ERR_INVALID_ARG;
    if (tile < 0 || tile >= tiles_m * tiles_n) return GEMM_ERR_INVALID_ARG;
    dtg::tile_coord(tile, tiles_m, tiles_n, group_m, *tile_m, *tile_n);
    return GEMM_OK;
}

const char* gemm_status_string(gemm_status_t s)
{
    switch (s) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG: invalid argument";
    case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED: misaligned pointer/leading dimension or size too large";
    case GEMM_ERR_ARCH: return "GEMM_ERR_ARCH: device is not sm_103";
    case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA: CUDA call or kernel launch failed";
    case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT: device watchdog expired";
    default: return "unknown gemm_status_t";
    }
}

int32_t gemm_api_version(void) { return GEMM_API_VERSION; }

}  // extern "C"

// ---------------------------------------------------------------- allocation-free entry point
//
// gemm_run_noalloc serves callers that cannot allocate device memory (a host engine that
// owns all device memory, paths that cannot take the device synchronisation an allocation
// may imply, a process at its memory limit).  The GEMM kernel's only scratch -- the
// 16-byte watchdog record that a handle normally cudaMallocs -- lives in the file-scope
// array below instead.  Nothing here calls cudaMalloc, cudaFree or any allocating routine.
namespace {

constexpr size_t kNoallocScratchBytes = 256;                 // stated maximum
constexpr size_t kNoallocRecordBytes = 4 * sizeof(int32_t);  // what the kernel writes
constexpr int kNoallocMaxDevices = 64;

// One copy per device, kept until the process exits.  On the host this name is only a
// stand-in for the symbol; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoallocScratchBytes / sizeof(int32_t)];

struct NoallocDevice {
    std::once_flag once;
    gemm_status_t setup = GEMM_ERR_CUDA;
    int32_t* scratch = nullptr;  // device address of g_noalloc_scratch on this device
    DeviceState dev;
};

NoallocDevice g_noalloc_devices[kNoallocMaxDevices];

// Runs once per device, with that device current (the caller's current device).
void noalloc_setup(NoallocDevice& d, int device)
{
    int sms = 0;
    d.setup = query_device(device, &sms);
    if (d.setup != GEMM_OK) return;
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) {
        d.setup = GEMM_ERR_CUDA;
        return;
    }
    d.scratch = static_cast<int32_t*>(addr);
    d.dev.num_sms = sms;
    d.setup = GEMM_OK;
}

}  // namespace

extern "C" gemm_status_t gemm_run_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                                          int64_t lda, int64_t ldb, int64_t ldc, gemm_layout_t layout,
                                          gemm_dtype_t dtype, void* stream, int32_t* watchdog_info)
{
    const gemm_status_t v = validate_args(A, B, C, M, N, K, lda, ldb, ldc, layout, dtype);
    if (v != GEMM_OK) return v;
    if (kNoallocRecordBytes > kNoallocScratchBytes) return GEMM_ERR_UNSUPPORTED;  // scratch need above the maximum
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) return GEMM_ERR_CUDA;
    if (device < 0 || device >= kNoallocMaxDevices) return GEMM_ERR_UNSUPPORTED;
    NoallocDevice& d = g_noalloc_devices[device];
    std::call_once(d.once, [&] { noalloc_setup(d, device); });
    if (d.setup != GEMM_OK) return d.setup;
    if (watchdog_info) std::memset(watchdog_info, 0, kNoallocRecordBytes);
    if (M == 0 || N == 0) return GEMM_OK;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The record keeps the previous call's contents: clear it before this launch.
    if (cudaMemsetAsync(d.scratch, 0, kNoallocRecordBytes, s) != cudaSuccess) return GEMM_ERR_CUDA;
    const LaunchOptions defaults;
    const gemm_status_t st =
        launch_gemm(defaults, d.dev, nullptr, nullptr, d.scratch, A, B, C, M, N, K, lda, ldb, ldc, layout, dtype, s);
    if (st != GEMM_OK) return st;

    if (watchdog_info) {
        int32_t info[4] = {0, 0, 0, 0};
        if (cudaMemcpyAsync(info, d.scratch, kNoallocRecordBytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
            return GEMM_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return GEMM_ERR_CUDA;
        std::memcpy(watchdog_info, info, kNoallocRecordBytes);
        if (info[0] != 0) return GEMM_ERR_TIMEOUT;
    }
    return GEMM_OK;
}

// Persistent warp-specialised tcgen05 GEMM for sm_103a: C = A·B, fp16/bf16 (or E4M3/E5M2)
// in, fp32 accumulate in tensor memory (TMEM), fp16/bf16 out.
//
// Structure (the four steps of "张量缩并：mma 语法" -- fill, load, multiply, store -- with
// the load and the multiply on different warps so they overlap, which the same page
// names as the next step after its one-warp kernel):
//
//   warp 0        TMA producer: per K block, waits for a free ring stage, arms its "full"
//                 barrier with the byte count and issues the A and B tile loads.  Reads
//                 outside the tensor are zero-filled by the TMA unit ("NineToothed GEMM
//                 语法入门" §5: out-of-range reads contribute 0).
//   warp 1        MMA issuer (one thread): per K block (128 bytes of K), four tcgen05.mma of
//                 32 bytes of K each into the TMEM accumulator (kind::f16 for 16-bit operands,
//                 kind::f8f6f4 for 8-bit ones, kind::mxf8f6f4.block_scale for 8-bit ones with
//                 E8M0 scales, kind::f16 .sp -- two MMAs of 32 K -- for a 2:4-sparse A), then
//                 tcgen05.commit releases the stage; after the item's last K block a commit
//                 marks the accumulator full.  The first MMA of an item overwrites (the
//                 zero-filled accumulator of §2), later ones add.  Sparsity metadata arrives
//                 with the stage, block scales in a ring of their own (one load per block for
//                 kScGroup stages); the MMA thread waits until warp 6 has copied them into
//                 TMEM.
//   warp 6        block-scaled and sparse kernels only (side data): per K block, once the
//                 stage is in, tcgen05.cp of its scales or metadata into the stage's TMEM
//                 columns, then a commit the MMA thread waits on.
//   warps 2..5    epilogue: tcgen05.ld of the accumulator (each warp owns the 32 TMEM lanes
//                 of its lane quadrant), C = alpha * acc + beta * C, fp32 -> fp16/bf16
//                 round-to-nearest-even, staging in 128-byte-swizzled shared memory and a TMA
//                 store that drops elements outside M x N (§5: masked write-back); C may be
//                 stored column-major (the page's transposed store).
//
// The accumulator is double-buffered in TMEM (2 x BN fp32 columns), so the epilogue of one
// item overlaps the main loop of the next; the block-scaled and sparse kernels keep one
// accumulator (their side data takes the other TMEM columns) and read it whole into registers
// before storing, which hands it back to the MMA thread early.
//
// Clusters: CLUSTER = 1 (one CTA) or 2 (a CTA pair).
//
// CTA pairs (CLUSTER == 2): a cluster of two CTAs on two SMs computes a 256 x BN tile with
// tcgen05.mma.cta_group::2 (M = 256).  This is the two-warpgroup kernel of the same page
// (two workers share one B tile, each takes its own rows of A) moved to the SM level:
// CTA r loads rows [128 r, 128 r + 128) of the A tile and B rows/columns
// [r BN/2, (r + 1) BN/2) into its own shared memory; one thread of the leader CTA (rank 0)
// issues the pair MMA, which reads both CTAs' halves and writes each CTA's 128 accumulator
// rows into that CTA's TMEM.  Per SM this halves the shared-memory bytes of B per MMA.
//   full[s]      lives in the leader, armed with both CTAs' bytes; both CTAs' TMA loads
//                complete on it (.cta_group::2 loads may signal the peer's barrier).
//   empty[s], acc_full[b]  in both CTAs; each commit of the leader arrives on both.
//   acc_empty[b] lives in the leader and counts the epilogue warps of both CTAs.
//
// Work schedule ("NineToothed GEMM 语法入门" §4: output tiles are independent, the K loop
// of one tile needs a merge if it is split).  Tiles are numbered in a grouped raster order
// (tile_coord).  With W work units (CTAs, or CTA pairs) running at once, tiles
// [0, dp_tiles) are taken whole, unit u doing tiles u, u + W, ...; the K blocks of the
// remaining tiles are dealt out as W contiguous ranges (stream-K), so every unit does the
// same amount of work instead of a last wave running part-empty.  A unit whose range covers
// only part of a tile writes its fp32 partial sums to a workspace slot and counts itself
// in; the last part to arrive adds all parts in K order (deterministic, whatever the
// arrival order) and writes C.  No unit ever waits for another.
//
// Every mbarrier wait is bounded (a watchdog on %globaltimer): on expiry the waiting
// thread records the place in the device error word and raises the abort flag of its CTA
// (and of the peer CTA); all roles leave their loops; the producer then waits (bounded)
// for its in-flight loads, the MMA thread for its in-flight MMAs, the epilogue for its
// stores, and the TMEM is freed before the CTA exits.  No trap, no unbounded spin.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "sm103_ptx.cuh"

namespace dtg {

constexpr int kBM = 128;          // accumulator rows per CTA (one TMEM lane per row)
constexpr int kRowBytes = 128;    // K bytes per operand row of a ring stage (one 128-byte swizzle row)
constexpr int kThreads = 192;     // 6 warps
constexpr int kThreadsSide = 224; // block-scaled and 2:4-sparse kernels: a 7th warp copies each
                                  // stage's side data (scales, metadata) into TMEM
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kEpiWarp0 = 2;
constexpr int kEpiWarps = 4;
constexpr int kSideWarp = 6;      // block-scaled and 2:4-sparse kernels only
constexpr int kEpiCols = 64;                        // columns per staged TMA store box
constexpr int kStgBytes = 32 * kEpiCols * 2;        // one warp's 32 x 64 box, 4 KB
constexpr uint32_t kWaitSleepNs = 20000;           // longest single suspension of a waiting thread
constexpr int kEpiBarrier = 1;                      // named barrier of the 4 epilogue warps

// Operand element types: 0 fp16, 1 bf16 (tcgen05 kind::f16), 2 E4M3, 3 E5M2 (kind::f8f6f4),
// 4 E4M3 and 5 E5M2 with one E8M0 scale per 32 K elements of each row of A and column of B
// (kind::mxf8f6f4, block-scaled), 6 fp16 and 7 bf16 with A 2:4-sparse (kind::f16 .sp).
// A ring stage holds one 128-byte swizzle row of K per row of B, so the number of K elements
// per stage and per MMA (32 bytes of B) depends on the element size; the shared-memory layout,
// the descriptors' byte offsets and the stage sizes do not.  A sparse A keeps half of K: its
// stage rows are 64 bytes (64-byte swizzle), and one sparse MMA covers 32 K (64 bytes of B).
template <int IN>
struct Operand {
    static constexpr bool kSparse = IN >= 6;
    static constexpr bool kF8 = IN >= 2 && IN < 6;
    static constexpr bool kMX = IN == 4 || IN == 5;  // block-scaled
    static constexpr int kBytes = kF8 ? 1 : 2;
    static constexpr int kStageK = 128 / kBytes;     // K elements per ring stage
    static constexpr int kMmaK = (kSparse ? 64 : 32) / kBytes;  // K elements per tcgen05.mma
    static constexpr int kNBlock = 128 / kBytes;     // N elements per 128-byte row of an N-major B box
    static constexpr int kAStageK = kSparse ? kStageK / 2 : kStageK;  // stored A elements per stage row
    static constexpr int kARowBytes = kAStageK * kBytes;
    static constexpr uint32_t kFormat = kSparse ? IN - 6 : (kF8 ? (IN - 2) & 1 : IN);  // A/B format
};

// Block scales travel in 512-byte chunks: the E8M0 exponents of 128 rows (of A, or columns
// of B) for 4 consecutive 32-long K blocks, i.e. one ring stage of 128 K elements.  Inside a
// chunk, row r and K block c sit at byte (r % 32) * 16 + (r / 32) * 4 + c, so that the 32
// 16-byte lines, copied into TMEM lanes 0-31 (and replicated into the other lane quadrants),
// put row r's four exponents in column r / 32 of lane r.  Chunk (row block rb, K group g) of
// a matrix with G = ceil(K / 128) K groups starts at byte (rb * G + g) * 512.
constexpr int kSfChunkBytes = 512;
constexpr int kSfChunkRows = 128;
// The chunks of kScGroup consecutive K groups of one row block are contiguous, so the producer
// loads a block's scales for kScGroup stages at once (one box per block instead of one per
// stage) into a ring of kScSlots slots of its own.
constexpr int kScGroup = 4;
constexpr int kScSlots = 2;
constexpr int kSfTmemCol = 256;  // first TMEM column of the per-stage side data (after one 256-column accumulator)
// CTA-pair kernels load side data (scale chunks, metadata chunks) through tensor maps that view
// the chunked buffer as rows of this many bytes, so a chunk is a box of whole rows.
constexpr int kSideRowBytes = 128;

// 2:4 sparsity metadata travels in 4096-byte chunks: 128 rows of A by one ring stage (64 K).
// The chunk holds one 2048-byte half per MMA of the stage (K [0, 32) and [32, 64) of the
// stage); in a half, TMEM lane l's 16 bytes (at l * 16) are its 32-bit metadata word followed
// by three padding words.  A group of four K elements takes 4 bits: the positions of its two
// kept elements (low two bits, then high two).  The MMA reads rows in pairs: for rows
// r = 16 b + i and r + 8 (i < 8), lane r holds groups 0-3 of the MMA's 32 K of row r (bits
// 0-15) and of row r + 8 (bits 16-31); lane r + 8 holds groups 4-7 of the two rows the same
// way (found by probing the instruction with single kept elements).  Chunk (row block rb,
// stage s) of a matrix with S = ceil(K / 64) stages starts at byte (rb * S + s) * 4096.  Each
// half goes to its own 8-column-aligned block of TMEM columns.
constexpr int kMetaChunkBytes = 4096;
constexpr int kMetaHalfBytes = 2048;
constexpr int kMetaTmemStride = 8;  // TMEM columns between the metadata of consecutive MMAs

// Error-word roles.
constexpr int kRoleProducer = 0, kRoleMma = 1, kRoleEpilogue = 2, kRoleDrain = 3, kRoleSide = 4;

struct KernelParams {
    int32_t M, N, K;
    int32_t tiles_m, tiles_n, num_kb, num_tiles;
    int32_t group_m;             // raster group (tile rows)
    int32_t fault_inject;        // test hook, see GEMM_OPT_FAULT_INJECT
    uint64_t timeout_ns;         // watchdog per wait
    int32_t* err;                // device error word [4]
    void* C;                     // output base, for the ragged-N edge written without TMA
    int64_t ldc;                 // output row pitch (elements)
    // stream-K schedule (dp_tiles == num_tiles: every tile whole, no workspace used)
    int32_t dp_tiles;            // tiles [0, dp_tiles) are done whole, round robin
    int64_t sk_base, sk_extra;   // K-block ranges over the rest: the first sk_extra units
                                 // take sk_base + 1 blocks, the others sk_base
    float* ws;                   // partial sums: [2 * units][ranks][BN / 4][128] float4
    int32_t* counters;           // arrivals per stream-K tile and CTA rank (kept at zero)
    // epilogue: C = alpha * A·B + beta * C (C read only when beta != 0); C stored row-major,
    // or column-major (C[m, n] at C + n * ldc + m) with c_col_major
    float alpha, beta;
    int32_t c_col_major;
    // block scales (kind::mxf8f6f4 kernels only): chunked as kSfChunkBytes describes
    int32_t sfb_blocks;          // ceil(N / 128)
    const uint8_t* sfa;          // ceil(M / 128) x num_kb chunks
    const uint8_t* sfb;          // sfb_blocks x num_kb chunks
    // 2:4 sparsity metadata (sparse kernels only): ceil(M / 128) x num_kb chunks of kMetaChunkBytes
    const uint8_t* meta;
    // 1: every second work item of a unit walks its K blocks backwards (not in block-scaled
    // kernels), so a wave of items starts on the A and B data the previous wave touched last
    int32_t k_snake;
};

// Linear tile index -> (tile row, tile column).  Tiles are taken in groups of group_m
// tile rows; inside a group the row index runs fastest, so CTAs that run at the same
// time share B tiles (same column) and a few A tiles, which keeps them in L2.
__host__ __device__ __forceinline__ void tile_coord(int64_t t, int64_t tiles_m, int64_t tiles_n,
                                                    int64_t group_m, int64_t& tm, int64_t& tn)
{
    const int64_t per_group = group_m * tiles_n;
    const int64_t g = t / per_group;
    const int64_t first_m = g * group_m;
    const int64_t rows = (tiles_m - first_m) < group_m ? (tiles_m - first_m) : group_m;
    const int64_t r = t - g * per_group;
    tm = first_m + r % rows;
    tn = r / rows;
}

// First stream-K K-block (relative to the stream-K region) of work unit u.
__host__ __device__ __forceinline__ int64_t sk_start(int64_t sk_base, int64_t sk_extra, int64_t u)
{
    return u * sk_base + (u < sk_extra ? u : sk_extra);
}

// Work unit whose stream-K range holds K-block x of the stream-K region.
__host__ __device__ __forceinline__ int64_t sk_owner(int64_t sk_base, int64_t sk_extra, int64_t x)
{
    const int64_t big = sk_extra * (sk_base + 1);
    return x < big ? x / (sk_base + 1) : sk_extra + (x - big) / sk_base;
}

// The work items of one unit, in order: (tile, first K block, end K block).  With k_snake,
// every second item (the 2nd, 4th, ... of the unit) is walked from its last K block down.
struct WorkIter {
    int64_t next_dp, step, u, u_end;
    int64_t count = 0;  // items returned so far

    __device__ __forceinline__ WorkIter(const KernelParams& p, int64_t unit, int64_t units)
        : next_dp(unit), step(units), u(0), u_end(0)
    {
        if (p.dp_tiles < p.num_tiles) {
            u = sk_start(p.sk_base, p.sk_extra, unit);
            u_end = sk_start(p.sk_base, p.sk_extra, unit + 1);
        }
    }

    __device__ __forceinline__ bool next(const KernelParams& p, int64_t& tile, int& kb0, int& kb1)
    {
        if (next_dp < p.dp_tiles) {
            tile = next_dp;
            kb0 = 0;
            kb1 = p.num_kb;
            next_dp += step;
            ++count;
            return true;
        }
        if (u < u_end) {
            const int64_t tr = u / p.num_kb;
            kb0 = static_cast<int>(u - tr * p.num_kb);
            const int64_t end = kb0 + (u_end - u);
            kb1 = static_cast<int>(end < p.num_kb ? end : p.num_kb);
            tile = p.dp_tiles + tr;
            u += kb1 - kb0;
            ++count;
            return true;
        }
        return false;
    }

    // Whether the item next() returned last is walked from its last K block down.
    __device__ __forceinline__ bool reversed(const KernelParams& p) const { return p.k_snake && (count & 1) == 0; }
};

// SF_BYTES: side-data bytes per ring stage (sparsity metadata; 0 without); SC_BYTES: bytes of
// one slot of the block-scale ring (kScSlots slots; 0 without); STG_BUFS: staging buffers per
// epilogue warp; A_ROW_BYTES: bytes of an A row per stage.
template <int B_ROWS, int STAGES, int SF_BYTES = 0, int STG_BUFS = 2, int A_ROW_BYTES = kRowBytes, int SC_BYTES = 0>
struct Smem {
    static constexpr int kABytes = kBM * A_ROW_BYTES;
    static constexpr int kBBytes = B_ROWS * kRowBytes;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kRing = STAGES * kStageBytes;
    static constexpr int kSfOff = kRing;
    static constexpr int kSfBytes = SF_BYTES;
    static constexpr int kScOff = kSfOff + STAGES * SF_BYTES;
    static constexpr int kScBytes = SC_BYTES;
    static constexpr int kStgOff = (kScOff + kScSlots * SC_BYTES + 1023) / 1024 * 1024;
    static constexpr int kStgBufs = STG_BUFS;
    static constexpr int kStg = kEpiWarps * STG_BUFS * kStgBytes;
    static constexpr int kBarOff = kStgOff + kStg;
    // full, empty, acc_full[2], acc_empty[2], drain, side-data-in-TMEM per stage, side-copy
    // drain, scale-ring full and empty per slot
    static constexpr int kNumBars = 3 * STAGES + 6 + 2 * kScSlots;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kTotal = kMiscOff + 16;     // tmem slot, abort flag, stream-K "last" flag
    static constexpr int kAlloc = kTotal + 1024;     // slack for aligning the base to 1 KB
    static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0 && kStageBytes % 1024 == 0,
                  "swizzle atoms need 1 KB alignment");
    static_assert(kStgOff % 1024 == 0, "the swizzled staging buffers need 1 KB alignment");
};

// Shared-memory layout of a kernel instantiation (host and device agree through this).
// Block-scaled kernels add a ring of scale slots (each the scale chunks of kScGroup stages:
// one chunk for A, one per 128 B rows, per stage) and, to stay within 227 KB, keep one staging
// buffer per epilogue warp; sparse kernels add the stage's metadata chunk and store A rows of
// 64 bytes (the CTA-pair sparse kernel also keeps one staging buffer, for a deeper ring).
template <int BN, int STAGES, int IN, bool PAIR>
struct KernelLayout {
    static constexpr int kBRows = BN / (PAIR ? 2 : 1);
    static constexpr bool kMX = Operand<IN>::kMX;
    static constexpr bool kSparse = Operand<IN>::kSparse;
    // Block-scale chunks per CTA and stage: its A rows' chunk and the B chunks of the whole tile
    // (each CTA of a pair produces all BN columns of its rows, so it holds every column's scales).
    static constexpr int kSfChunks = kMX ? 1 + BN / kSfChunkRows : 0;
    static constexpr int kSfBytes = kSparse ? kMetaChunkBytes : 0;
    static constexpr int kScBytes = kSfChunks * kScGroup * kSfChunkBytes;
    using S = Smem<kBRows, STAGES, kSfBytes, (kMX || (kSparse && PAIR)) ? 1 : 2, Operand<IN>::kARowBytes, kScBytes>;
};

// tcgen05 shared-memory matrix descriptor for a 128-byte-swizzled operand tile.
//   bits  0-13 start address >> 4        bits 16-29 leading-dimension byte offset >> 4
//   bits 32-45 stride-dimension offset >> 4   bits 46-47 fixed 0b01
//   bits 49-51 base offset (0: tiles are 1 KB aligned)   bits 61-63 layout (2 = 128B swizzle)
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// tcgen05 shared-memory matrix descriptor for an unswizzled matrix of 16-byte rows: core
// matrices of 8 rows x 16 B (128 contiguous bytes), 8-row groups `sbo` bytes apart.
__device__ __forceinline__ uint64_t smem_desc_plain(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;  // layout bits 61-63 = 0: no swizzle
    return d;
}

// tcgen05 shared-memory matrix descriptor for a 64-byte-swizzled K-major operand tile (rows of
// 64 bytes, 8-row atoms of 512 bytes `sbo` apart).
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 4ull << 61;  // layout: 64-byte swizzle
    return d;
}

// Instruction descriptor of tcgen05.mma.kind::mxf8f6f4.block_scale: D fp32 (implied), A and
// B of the same 8-bit format (0 E4M3, 1 E5M2), A K-major, B K-major or N-major, scale format
// E8M0 (bit 23), M x N shape.  Bits 29-30 / 4-5 select the byte of the TMEM words holding
// the scales of A / B: mx_scale_ids(k) for the k-th 32-long K block of a stage.
template <uint32_t FORMAT, bool B_MN_MAJOR, int M, int N>
__host__ __device__ constexpr uint32_t idesc_mx()
{
    return (FORMAT << 7) | (FORMAT << 10) | ((B_MN_MAJOR ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) | (static_cast<uint32_t>(M >> 4) << 24);
}

__host__ __device__ constexpr uint32_t mx_scale_ids(uint32_t k) { return (k << 29) | (k << 4); }

// Instruction descriptor of tcgen05.mma.kind::f16 / kind::f8f6f4: D fp32, A and B of the same
// format (kind::f16: 0 fp16, 1 bf16; kind::f8f6f4: 0 E4M3, 1 E5M2), A K-major, B K-major (TN)
// or N-major (NN), M x N shape.
template <uint32_t FORMAT, bool B_MN_MAJOR, int M, int N>
__host__ __device__ constexpr uint32_t idesc_mma()
{
    return (1u << 4)                                  // D format: f32
           | (FORMAT << 7)                            // A format
           | (FORMAT << 10)                           // B format
           | ((B_MN_MAJOR ? 1u : 0u) << 16)           // B major-ness
           | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

struct Watchdog {
    volatile int32_t* abort_flag;  // shared memory
    const KernelParams* p;
    uint32_t peer_abort = 0;  // shared::cluster address of the peer CTA's flag (CTA pair), 0 = none

    __device__ __forceinline__ void fail(int role, int64_t tile, int kb) const
    {
        *abort_flag = 1;
        if (peer_abort) ptx::st_shared_cluster_u32(peer_abort, 1u);
        if (atomicCAS(p->err, 0, 1) == 0) {
            p->err[1] = role;
            p->err[2] = static_cast<int32_t>(blockIdx.x);
            p->err[3] = static_cast<int32_t>(tile * 65536 + kb);
        }
    }

    // Wait for the phase of parity `parity` of `bar`.  False if the CTA is aborting or
    // this wait ran past the limit (then the failure is recorded).
    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, int role, int64_t tile,
                                         int kb) const
    {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = ptx::globaltimer_ns();
        for (;;) {
            // Sleep until the phase completes (or kWaitSleepNs passes): a waiting warp must
            // not take issue slots from the producer and MMA warps on its scheduler.
            if (ptx::mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
            if (*abort_flag) return false;
            if (ptx::globaltimer_ns() - t0 > p->timeout_ns) {
                fail(role, tile, kb);
                return false;
            }
        }
    }

    // Bounded wait that ignores the abort flag: used while draining in-flight work.
    __device__ __forceinline__ bool drain(uint32_t bar, uint32_t parity) const
    {
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(bar, parity)) {
            if (ptx::globaltimer_ns() - t0 > p->timeout_ns) {
                fail(kRoleDrain, -1, 0);
                return false;
            }
        }
        return true;
    }
};

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(uint32_t lo_bits, uint32_t hi_bits)
{
    const float lo = __uint_as_float(lo_bits), hi = __uint_as_float(hi_bits);
    if constexpr (BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

template <bool BF16>
__device__ __forceinline__ float load16(const uint16_t* src)
{
    const uint16_t b = *src;
    if constexpr (BF16)
        return __bfloat162float(__ushort_as_bfloat16(b));
    else
        return __half2float(__ushort_as_half(b));
}

template <bool BF16>
__device__ __forceinline__ uint16_t cvt16(uint32_t f_bits)
{
    if constexpr (BF16)
        return __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(f_bits)));
    else
        return __half_as_ushort(__float2half_rn(__uint_as_float(f_bits)));
}

// C = alpha * acc + beta * C on the 32-row x 64-column box of C at (row y, column x) that
// this warp holds (lane = row, v = the 64 fp32 accumulator bit patterns of that row, scaled
// in place).  "张量缩并：mma 语法" states the contraction as C += A × B (alpha = beta = 1);
// the existing C is read only when beta != 0.
template <bool BF16>
__device__ __forceinline__ void scale_box(uint32_t (&v)[64], int32_t x, int32_t y, int lane, const KernelParams& p)
{
    const int64_t row = static_cast<int64_t>(y) + lane;  // this thread's output row m
    if (p.alpha != 1.0f || p.beta != 0.0f) {
        const uint16_t* c16 = static_cast<const uint16_t*>(p.C);
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            float f = p.alpha * __uint_as_float(v[i]);
            const int64_t col = static_cast<int64_t>(x) + i;
            if (p.beta != 0.0f && row < p.M && col < p.N)
                f = fmaf(p.beta, load16<BF16>(p.c_col_major ? c16 + col * p.ldc + row : c16 + row * p.ldc + col),
                         f);
            v[i] = __float_as_uint(f);
        }
    }
}

// Round the 64 fp32 values of a box row to 16 bits (round to nearest even), two per word:
// element 2i in the low half of h[i].
template <bool BF16>
__device__ __forceinline__ void pack_box(const uint32_t (&v)[64], uint32_t (&h)[32])
{
#pragma unroll
    for (int i = 0; i < 32; ++i) h[i] = pack2<BF16>(v[2 * i], v[2 * i + 1]);
}

__device__ __forceinline__ uint16_t half_of(const uint32_t (&h)[32], int i)
{
    return static_cast<uint16_t>((h[i >> 1] >> ((i & 1) * 16)) & 0xFFFFu);
}

// Write a box of C already rounded to 16 bits (h, as pack_box leaves it).
//  * Row-major C: the box goes through a 128-byte-swizzled staging buffer and one TMA store,
//    which drops rows >= M and columns >= N (the masked write-back of "NineToothed GEMM 语法
//    入门" §5).  A TMA store clips the inner dimension only to 16-byte granules, so when N
//    is not a multiple of 8 the box that straddles column N is written with plain masked
//    stores instead.
//  * Column-major C (the transposed store of "张量缩并：mma 语法", mma.store.transp): the box
//    is staged transposed (64 rows of n, 32 m values each) and stored through a tensor map of
//    C's storage; a box straddling a ragged M (M % 8 != 0) is written with plain stores.
// STG_BUFS: staging buffers of this warp (1 or 2).  Returns true if the staging buffer was
// used (the caller then moves on to its next buffer).
template <int STG_BUFS>
__device__ __forceinline__ bool store_packed(const uint32_t (&h)[32], int32_t x, int32_t y, int lane, uint32_t stg,
                                             const CUtensorMap* tmC, const KernelParams& p)
{
    const int64_t row = static_cast<int64_t>(y) + lane;  // this thread's output row m
    if (p.c_col_major) {
        if ((p.M & 7) != 0 && y + 32 > p.M) {
            if (row < p.M) {
                uint16_t* c16 = static_cast<uint16_t*>(p.C);
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if (x + i < p.N) c16[static_cast<int64_t>(x + i) * p.ldc + row] = half_of(h, i);
            }
            return false;
        }
        if (lane == 0) ptx::bulk_wait_group_read<STG_BUFS - 1>();
        __syncwarp();
        // Dense staging box: (n, m) at n * 64 B + m * 2 B.
#pragma unroll
        for (int i = 0; i < 64; ++i)
            asm volatile("st.shared.u16 [%0], %1;" ::"r"(stg + i * 64 + lane * 2), "h"(half_of(h, i)) : "memory");
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            if (x < p.N && y < p.M) ptx::tma_store_2d(tmC, stg, y, x);
            ptx::bulk_commit_group();
        }
        return true;
    }
    if ((p.N & 7) != 0 && x + kEpiCols > p.N) {
        if (row < p.M && x < p.N) {
            uint16_t* crow = static_cast<uint16_t*>(p.C) + row * p.ldc;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                const int32_t col = x + ch * 8;
                if (col + 8 <= p.N) {  // a whole 16-byte chunk: one vector store
                    *reinterpret_cast<uint4*>(crow + col) = make_uint4(h[4 * ch], h[4 * ch + 1], h[4 * ch + 2],
                                                                       h[4 * ch + 3]);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (col + e < p.N) crow[col + e] = half_of(h, 8 * ch + e);
                }
            }
        }
        return false;
    }
    // The staging buffer is reusable once the store issued from it STG_BUFS boxes ago has
    // finished reading it.
    if (lane == 0) ptx::bulk_wait_group_read<STG_BUFS - 1>();
    __syncwarp();
    const uint32_t srow = stg + lane * 128;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        // 16-byte chunk ch of this row lands at chunk (ch ^ row%8): the 128-byte swizzle
        // the TMA store expects.
        const uint32_t addr = srow + ((ch ^ (lane & 7)) << 4);
        ptx::st_shared_v4(addr, h[4 * ch], h[4 * ch + 1], h[4 * ch + 2], h[4 * ch + 3]);
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (x < p.N && y < p.M) ptx::tma_store_2d(tmC, stg, x, y);
        ptx::bulk_commit_group();
    }
    return true;
}

// scale_box, pack_box and store_packed in one: the box of fp32 accumulator values v.
template <bool BF16, int STG_BUFS>
__device__ __forceinline__ bool store_box(uint32_t (&v)[64], int32_t x, int32_t y, int lane, uint32_t stg,
                                          const CUtensorMap* tmC, const KernelParams& p)
{
    scale_box<BF16>(v, x, y, lane, p);
    uint32_t h[32];
    pack_box<BF16>(v, h);
    return store_packed<STG_BUFS>(h, x, y, lane, stg, tmC, p);
}

__device__ __forceinline__ void epilogue_bar_sync()
{
    asm volatile("bar.sync %0, %1;" ::"n"(kEpiBarrier), "n"(kEpiWarps * 32) : "memory");
}

// Barrier of the 4 epilogue warps that also ANDs a flag over their 128 threads: the
// epilogue warps use it to agree on leaving their loop, so they always execute the same
// iterations (and therefore the same named barriers).
__device__ __forceinline__ bool epilogue_bar_and(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.and.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}\n"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "n"(kEpiBarrier), "n"(kEpiWarps * 32)
        : "memory");
    return r != 0;
}

// Stream-K bookkeeping for stream-K tile tr (relative to the stream-K region): the first
// unit with a part of it and the number of parts.
__device__ __forceinline__ void sk_parts(const KernelParams& p, int64_t tr, int64_t& first_unit, int64_t& parts)
{
    first_unit = sk_owner(p.sk_base, p.sk_extra, tr * p.num_kb);
    parts = sk_owner(p.sk_base, p.sk_extra, (tr + 1) * p.num_kb - 1) - first_unit + 1;
}

// Workspace slot of unit u's part of stream-K tile tr: each unit has two slots, for the
// tile its range starts in (0) and the tile it ends in (1).
__device__ __forceinline__ int64_t sk_slot(const KernelParams& p, int64_t u, int64_t tr)
{
    return u * 2 + (sk_start(p.sk_base, p.sk_extra, u) >= tr * p.num_kb ? 0 : 1);
}

// IN: operand type (see Operand); OUT_BF16: C is bf16 (else fp16).  CLUSTER: 1 (one CTA) or 2
// (a CTA pair).  tmS, tmS2: the side data
// of a CTA-pair kernel seen as rows of kSideRowBytes -- the metadata chunks (sparse), or the A and
// the B scale chunks (block-scaled); unused otherwise.
template <int BN, int STAGES, int IN, bool OUT_BF16, bool NN, int CLUSTER>
__global__ void __launch_bounds__((Operand<IN>::kMX || Operand<IN>::kSparse) ? kThreadsSide : kThreads, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmS,
                        const __grid_constant__ CUtensorMap tmS2, const KernelParams p)
{
    using T = Operand<IN>;
    static_assert(CLUSTER == 1 || CLUSTER == 2, "one CTA or a CTA pair");
    constexpr bool PAIR = CLUSTER == 2;
    constexpr int kRanks = PAIR ? 2 : 1;       // CTAs per MMA (pair)
    constexpr int kTileM = kBM * kRanks;       // output rows per tile
    constexpr int kBRows = BN / kRanks;        // B rows (TN) / columns (NN) this CTA loads
    static_assert(BN == 64 || BN == 128 || BN == 256, "one MMA of N = BN per K step");
    static_assert(!NN || kBRows % T::kNBlock == 0, "an N-major B box is one 128-byte row of N");
    // Block-scaled and sparse kernels keep one accumulator and put the side data of every
    // ring stage (scales, metadata) in the TMEM columns after it; the others double-buffer
    // the accumulator.
    constexpr bool kSide = T::kMX || T::kSparse;
    constexpr int kAccBufs = kSide ? 1 : 2;
    constexpr uint32_t kTmemCols = kSide ? 512 : 2 * BN;
    static_assert(kTmemCols == 128 || kTmemCols == 256 || kTmemCols == 512, "TMEM allocations are powers of two");
    using L = typename KernelLayout<BN, STAGES, IN, PAIR>::S;
    constexpr int kSfChunks = KernelLayout<BN, STAGES, IN, PAIR>::kSfChunks;  // block-scale chunks per stage: A, then B
    constexpr int kSideCols = T::kMX ? kSfChunks * 4 : (T::kSparse ? 2 * kMetaTmemStride : 0);  // TMEM cols / stage
    static_assert(!kSide || (BN <= kSfTmemCol &&
                             kSfTmemCol + STAGES * kSideCols <= static_cast<int>(kTmemCols)),
                  "the accumulator and the side data fit in TMEM");

    extern __shared__ uint8_t smem_raw[];
    // Align the working area to 1 KB (128-byte swizzle atoms repeat every 8 rows).
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* const smem = smem_raw + (base - raw_addr);

    const uint32_t bar0 = base + L::kBarOff;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
    auto sfr_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + 5 + s); };  // side data of stage s in TMEM
    const uint32_t sdrain_bar = bar0 + 8u * (3 * STAGES + 5);
    auto scf_bar = [&](int q) { return bar0 + 8u * (3 * STAGES + 6 + q); };             // scale slot q loaded
    auto sce_bar = [&](int q) { return bar0 + 8u * (3 * STAGES + 6 + kScSlots + q); };  // scale slot q free
    uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    volatile int32_t* const abort_flag = reinterpret_cast<volatile int32_t*>(smem + L::kMiscOff + 4);
    volatile int32_t* const last_flag = reinterpret_cast<volatile int32_t*>(smem + L::kMiscOff + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t crank = PAIR ? ptx::cluster_ctarank() : 0u;  // rank in the pair; 0: the leader (issues its MMAs)
    const uint32_t rank = crank;
    const bool leader = rank == 0;
    const int64_t unit = PAIR ? static_cast<int64_t>(ptx::cluster_id_x()) : static_cast<int64_t>(blockIdx.x);
    const int64_t units = PAIR ? static_cast<int64_t>(ptx::num_clusters_x()) : static_cast<int64_t>(gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(accf_bar(b), 1);
            ptx::mbar_init(acce_bar(b), kEpiWarps * kRanks);
        }
        ptx::mbar_init(drain_bar, 1);
        if constexpr (kSide) {
            for (int s = 0; s < STAGES; ++s) ptx::mbar_init(sfr_bar(s), 1);
            ptx::mbar_init(sdrain_bar, 1);
            if constexpr (T::kMX)
                for (int q = 0; q < kScSlots; ++q) {
                    ptx::mbar_init(scf_bar(q), 1);
                    ptx::mbar_init(sce_bar(q), 1);
                }
        }
        *abort_flag = 0;
        *last_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
        ptx::prefetch_tmap(&tmC);
        if constexpr (T::kSparse && PAIR) ptx::prefetch_tmap(&tmS);
        if constexpr (T::kMX) {
            ptx::prefetch_tmap(&tmS);
            ptx::prefetch_tmap(&tmS2);
        }
    }
    if (warp == kMmaWarp) {
        if constexpr (PAIR) {
            ptx::tmem_alloc_pair(ptx::smem_addr(tmem_slot), kTmemCols);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
            ptx::tmem_relinquish();
        }
    }
    ptx::tc_fence_before_sync();
    if constexpr (PAIR)
        ptx::cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
    else
        __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // Everything above touched only shared memory, TMEM and the kernel's parameters; global
    // memory (A, B, C, side data, workspace) waits for the stream's previous kernel.
    ptx::grid_dependency_wait();
    ptx::launch_dependents();

    Watchdog wd{abort_flag, &p};
    if constexpr (PAIR) {
        const uint32_t own = ptx::smem_addr(const_cast<int32_t*>(abort_flag));
        wd.peer_abort = ptx::mapa_shared(own, crank ^ 1u);
    }

    if (warp == kProducerWarp) {
        if (lane == 0) {
            // ---------------------------------------------------------------- producer
            uint32_t armed_mask = 0, armed_parity = 0;  // leader: stages armed, last parity
            uint32_t sc_armed_mask = 0, sc_armed_parity = 0;  // leader: scale slots armed, last parity
            int stage = 0;
            uint32_t phase = 0;
            int sc_slot = 0;  // block-scale ring
            uint32_t sc_phase = 0;
            int64_t loaded = 0;
            WorkIter it(p, unit, units);
            int64_t tile;
            int kb0, kb1;
            while (it.next(p, tile, kb0, kb1)) {
                int64_t tm, tn;
                tile_coord(tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
                const int32_t y_a = static_cast<int32_t>(tm * kTileM + rank * kBM);
                const int32_t n_b = static_cast<int32_t>(tn * BN + rank * kBRows);
                // Block scales: the A chunk of this tile row and the B chunks of this tile's
                // columns that exist (a ragged N may leave out the last).
                int sf_b_chunks = 0;
                if constexpr (T::kMX) {
                    const int64_t nb0 = tn * (BN / kSfChunkRows);
                    sf_b_chunks = static_cast<int>(p.sfb_blocks - nb0);
                    if (sf_b_chunks > kSfChunks - 1) sf_b_chunks = kSfChunks - 1;
                }
                const bool rev = !T::kMX && it.reversed(p);
                for (int i = 0; i < kb1 - kb0; ++i, ++loaded) {
                    const int kb = rev ? kb1 - 1 - i : kb0 + i;  // the i-th K block this item loads
                    if (!wd.wait(empty_bar(stage), phase ^ 1u, kRoleProducer, tile, kb)) goto producer_done;
                    if constexpr (T::kMX) {
                        // Every kScGroup stages of an item: the scale chunks of those stages, one
                        // box of kScGroup chunks per block (A's, then B's), into the next slot of
                        // the scale ring, completing on that slot's barrier in the leader.
                        if (i % kScGroup == 0) {
                            if (!wd.wait(sce_bar(sc_slot), sc_phase ^ 1u, kRoleProducer, tile, kb)) goto producer_done;
                            const uint32_t sc = base + L::kScOff + sc_slot * L::kScBytes;
                            const uint32_t scb = PAIR ? ptx::mapa_shared(scf_bar(sc_slot), 0u) : scf_bar(sc_slot);
                            if (leader) {
                                ptx::mbar_arrive_expect_tx(scf_bar(sc_slot),
                                                           kRanks * (1 + sf_b_chunks) * kScGroup * kSfChunkBytes);
                                sc_armed_mask |= 1u << sc_slot;
                                sc_armed_parity = (sc_armed_parity & ~(1u << sc_slot)) | (sc_phase << sc_slot);
                            }
                            auto load_sc = [&](uint32_t dst, const CUtensorMap* tm_, int64_t chunk) {
                                const int32_t y = static_cast<int32_t>(chunk * (kSfChunkBytes / kSideRowBytes));
                                if constexpr (PAIR)
                                    ptx::tma_load_2d_pair(dst, tm_, 0, y, scb);
                                else
                                    ptx::tma_load_2d(dst, tm_, 0, y, scb);
                            };
                            const int64_t nb0 = tn * (BN / kSfChunkRows);
                            load_sc(sc, &tmS, (tm * kRanks + rank) * p.num_kb + kb);
                            for (int j = 0; j < sf_b_chunks; ++j)
                                load_sc(sc + (1 + j) * (kScGroup * kSfChunkBytes), &tmS2, (nb0 + j) * p.num_kb + kb);
                        }
                    }
                    if (p.fault_inject && unit == 0 && loaded == 1) {
                        // Test hook: every CTA of the first unit leaves this stage unloaded (and
                        // the leader leaves it unarmed), so the MMA thread's wait on it runs out
                        // and the watchdog path is exercised with no load of that stage in flight.
                    } else {
                        const uint32_t sa = base + stage * L::kStageBytes;
                        const uint32_t sb = sa + L::kABytes;
                        const int32_t k0 = kb * T::kStageK;
                        const uint32_t fb = PAIR ? ptx::mapa_shared(full_bar(stage), 0u) : full_bar(stage);
                        if (leader) {
                            const int sf_bytes = T::kSparse ? kMetaChunkBytes : 0;
                            ptx::mbar_arrive_expect_tx(full_bar(stage), kRanks * (L::kStageBytes + sf_bytes));
                            armed_mask |= 1u << stage;
                            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                        }
                        auto load = [&](uint32_t dst, const CUtensorMap* tm_, int32_t x, int32_t y) {
                            if constexpr (PAIR)
                                ptx::tma_load_2d_pair(dst, tm_, x, y, fb);
                            else
                                ptx::tma_load_2d(dst, tm_, x, y, fb);
                        };
                        load(sa, &tmA, kb * T::kAStageK, y_a);
                        if constexpr (NN) {
                            // B stored K x N: boxes of one 128-byte row of N (kNBlock elements)
                            // by kStageK rows of K, kStageK * 128 bytes each.
#pragma unroll
                            for (int q = 0; q < kBRows / T::kNBlock; ++q)
                                load(sb + q * (T::kStageK * 128), &tmB, n_b + q * T::kNBlock, k0);
                        } else {
                            // B stored N x K: one box of kStageK (K) x kBRows (N rows).
                            load(sb, &tmB, k0, n_b);
                        }
                        if constexpr (T::kSparse) {
                            // This CTA's 128 rows: metadata chunk (row block, stage) -- one 1-D bulk
                            // copy, or, in a pair, a TMA box of whole kSideRowBytes rows that completes
                            // on the leader's barrier like the A and B boxes.
                            const int64_t chunk = (tm * kRanks + rank) * p.num_kb + kb;
                            if constexpr (PAIR)
                                load(base + L::kSfOff + stage * L::kSfBytes, &tmS, 0,
                                     static_cast<int32_t>(chunk * (kMetaChunkBytes / kSideRowBytes)));
                            else
                                ptx::bulk_load_1d(base + L::kSfOff + stage * L::kSfBytes,
                                                  p.meta + chunk * kMetaChunkBytes, kMetaChunkBytes, fb);
                        }
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if constexpr (T::kMX) {
                        if (i % kScGroup == kScGroup - 1 || i == kb1 - kb0 - 1) {
                            if (++sc_slot == kScSlots) {
                                sc_slot = 0;
                                sc_phase ^= 1u;
                            }
                        }
                    }
                }
            }
            // Tail: wait (bounded) until the MMA thread has released every stage this
            // producer filled (and the side-data warp every scale slot), so no
            // tcgen05.commit arrival is still heading for this CTA's barriers when it leaves.
            for (int i = 0; i < STAGES; ++i) {
                if (!wd.wait(empty_bar(stage), phase ^ 1u, kRoleProducer, -1, i)) goto producer_done;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if constexpr (T::kMX) {
                for (int i = 0; i < kScSlots; ++i) {
                    if (!wd.wait(sce_bar(sc_slot), sc_phase ^ 1u, kRoleProducer, -1, i)) break;
                    if (++sc_slot == kScSlots) {
                        sc_slot = 0;
                        sc_phase ^= 1u;
                    }
                }
            }
        producer_done:
            // The leader's full barriers count every load of the CTA (pair): waiting on them
            // (bounded) covers every load still in flight.
            if (leader) {
                for (int s = 0; s < STAGES; ++s)
                    if (armed_mask & (1u << s)) wd.drain(full_bar(s), (armed_parity >> s) & 1u);
                if constexpr (T::kMX)
                    for (int q = 0; q < kScSlots; ++q)
                        if (sc_armed_mask & (1u << q)) wd.drain(scf_bar(q), (sc_armed_parity >> q) & 1u);
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0 && leader) {
            // ---------------------------------------------------------------- MMA issuer
            // Sparse MMAs: the dense descriptor with the sparsity flag (bit 2).
            constexpr uint32_t idesc = T::kMX ? idesc_mx<T::kFormat, NN, kTileM, BN>()
                                              : (idesc_mma<T::kFormat, NN, kTileM, BN>() | (T::kSparse ? 4u : 0u));
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool aborted = false;
            WorkIter it(p, unit, units);
            int64_t tile;
            int kb0, kb1;
            while (!aborted && it.next(p, tile, kb0, kb1)) {
                if (!wd.wait(acce_bar(acc), acc_phase ^ 1u, kRoleMma, tile, -1)) {
                    aborted = true;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                const bool rev = !T::kMX && it.reversed(p);
                for (int i = 0; i < kb1 - kb0; ++i) {
                    const int kb = rev ? kb1 - 1 - i : kb0 + i;
                    // Block-scaled and sparse kernels wait for the stage's side data to be in
                    // TMEM (the side warp copies it once the stage's data is in); the others
                    // for the stage's data.
                    if (!wd.wait(kSide ? sfr_bar(stage) : full_bar(stage), phase, kRoleMma, tile, kb)) {
                        aborted = true;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint32_t sa = base + stage * L::kStageBytes;
                    const uint32_t sb = sa + L::kABytes;
                    // Block scales of this stage in TMEM: A at sf_tmem, B from sf_tmem + 4.
                    uint32_t sf_tmem = 0;
                    if constexpr (T::kMX) sf_tmem = tmem_base + static_cast<uint32_t>(kSfTmemCol + stage * kSideCols);
                    // Sparsity metadata of this stage in TMEM: MMA k's at sf_tmem + 8 k.
                    if constexpr (T::kSparse) sf_tmem = tmem_base + static_cast<uint32_t>(kSfTmemCol + stage * kSideCols);
#pragma unroll
                    for (int k = 0; k < T::kStageK / T::kMmaK; ++k) {
                        // A (K-major): the k-th K slice starts 32 B further along each row;
                        // 128-byte-swizzled rows, 8-row groups 1 KB apart (SBO) -- or, for a
                        // sparse A, 64-byte-swizzled rows with 512-byte groups.
                        const uint64_t adesc =
                            T::kSparse ? smem_desc_sw64(sa + k * 32, 16, 512) : smem_desc_sw128(sa + k * 32, 16, 1024);
                        const uint32_t accumulate = (i != 0 || k != 0) ? 1u : 0u;  // the item's first MMA overwrites
                        uint64_t bdesc;
                        if constexpr (NN) {
                            // B (N-major): rows are K; the k-th slice starts kMmaK rows of 128 B
                            // on; 128-byte-wide N blocks are kStageK rows apart (LBO), 8-row K
                            // groups 1 KB apart (SBO).
                            bdesc = smem_desc_sw128(sb + k * (T::kMmaK * 128), T::kStageK * 128, 1024);
                        } else {
                            // B (K-major): the k-th slice starts kMmaK elements along each row.
                            bdesc = smem_desc_sw128(sb + k * (T::kMmaK * T::kBytes), 16, 1024);
                        }
                        if constexpr (PAIR) {
                            if constexpr (T::kMX)
                                ptx::mma_mxf8_pair(d_tmem, adesc, bdesc, idesc | mx_scale_ids(k), sf_tmem, sf_tmem + 4,
                                                   accumulate);
                            else if constexpr (T::kSparse)
                                ptx::mma_sp_f16_pair(d_tmem, adesc, bdesc, sf_tmem + k * kMetaTmemStride, idesc,
                                                     accumulate);
                            else if constexpr (T::kF8)
                                ptx::mma_f8_pair(d_tmem, adesc, bdesc, idesc, accumulate);
                            else
                                ptx::mma_f16_pair(d_tmem, adesc, bdesc, idesc, accumulate);
                        } else {
                            if constexpr (T::kMX)
                                ptx::mma_mxf8_cta1(d_tmem, adesc, bdesc, idesc | mx_scale_ids(k), sf_tmem, sf_tmem + 4,
                                                   accumulate);
                            else if constexpr (T::kSparse)
                                ptx::mma_sp_f16_cta1(d_tmem, adesc, bdesc, sf_tmem + k * kMetaTmemStride, idesc,
                                                     accumulate);
                            else if constexpr (T::kF8)
                                ptx::mma_f8_cta1(d_tmem, adesc, bdesc, idesc, accumulate);
                            else
                                ptx::mma_f16_cta1(d_tmem, adesc, bdesc, idesc, accumulate);
                        }
                    }
                    // The stage is free once these MMAs finish (in both CTAs of a pair).
                    if constexpr (PAIR)
                        ptx::mma_commit_pair(empty_bar(stage), 0x3);
                    else
                        ptx::mma_commit_cta1(empty_bar(stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (aborted) break;
                if constexpr (PAIR)
                    ptx::mma_commit_pair(accf_bar(acc), 0x3);  // accumulator complete
                else
                    ptx::mma_commit_cta1(accf_bar(acc));
                if (++acc == kAccBufs) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (aborted) {
                // Let every MMA issued so far finish before the TMEM is released.
                if constexpr (PAIR)
                    ptx::mma_commit_pair(drain_bar, static_cast<uint16_t>(1u << crank));
                else
                    ptx::mma_commit_cta1(drain_bar);
                wd.drain(drain_bar, 0);
            }
        }
        __syncwarp();
    } else if (kSide && warp == kSideWarp) {
        if (lane == 0 && leader) {
            // ---------------------------------------------------------------- side data
            // Block-scaled and sparse kernels: once a stage's data is in, its side data goes
            // from shared memory into the stage's TMEM columns -- the scale chunks (4 columns
            // each: A's, then B's) or the two metadata halves (one 8-column block per MMA) --
            // and a commit tells the MMA thread it is there.  Issued by the MMA thread itself,
            // these copies held its MMAs back (measured: three copies per stage cost ~15 % of
            // the tensor pipe's time); from this warp they overlap the MMAs.  The stage is
            // released (empty barrier) only after the MMAs that follow the copies, so no copy
            // outlives its source.  Block scales come from their own ring (a slot holds
            // kScGroup stages' chunks): a slot is released by a commit after the copies of its
            // last stage.
            int stage = 0;
            uint32_t phase = 0;
            int sc_slot = 0;
            uint32_t sc_phase = 0;
            bool aborted = false;
            WorkIter it(p, unit, units);
            int64_t tile;
            int kb0, kb1;
            while (!aborted && it.next(p, tile, kb0, kb1)) {
                const bool rev = !T::kMX && it.reversed(p);
                for (int i = 0; i < kb1 - kb0; ++i) {
                    const int kb = rev ? kb1 - 1 - i : kb0 + i;
                    const int pos = i % kScGroup;  // stage within its scale slot
                    if constexpr (T::kMX) {
                        if (pos == 0 && !wd.wait(scf_bar(sc_slot), sc_phase, kRoleSide, tile, kb)) {
                            aborted = true;
                            break;
                        }
                    }
                    // Copies wait for the whole stage (issued as soon as the stage's TMEM columns
                    // were free, they ran between the MMAs of the stage before and slowed them:
                    // 8192^3 E4M3 2880 against 3259 TF/s).
                    if (!wd.wait(full_bar(stage), phase, kRoleSide, tile, kb)) {
                        aborted = true;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint32_t col = static_cast<uint32_t>(kSfTmemCol + stage * kSideCols);
                    const uint32_t sf_tmem = tmem_base + col;
                    const uint32_t sf = base + L::kSfOff + stage * L::kSfBytes;
                    if constexpr (T::kMX) {
                        // Chunk c of this stage: block c's box in the slot, stage pos of kScGroup.
                        const uint32_t sc = base + L::kScOff + sc_slot * L::kScBytes + pos * kSfChunkBytes;
#pragma unroll
                        for (int c = 0; c < kSfChunks; ++c) {
                            const uint64_t d = smem_desc_plain(sc + c * (kScGroup * kSfChunkBytes), 0, 128);
                            if constexpr (PAIR)
                                ptx::tmem_cp_32x128b_warpx4_pair(sf_tmem + 4 * c, d);
                            else
                                ptx::tmem_cp_32x128b_warpx4(sf_tmem + 4 * c, d);
                        }
                    } else {
                        // Per MMA k, 128 rows x 16 bytes -> TMEM lanes 0-127, columns
                        // sf_tmem + 8k .. + 3 (8-column aligned).  The addresses are checked
                        // against that alignment; a violation is reported, not issued.
                        if ((col % kMetaTmemStride) != 0 || (sf & 127u) != 0) {
                            wd.fail(kRoleSide, tile, kb);
                            aborted = true;
                            break;
                        }
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint64_t d = smem_desc_plain(sf + h * kMetaHalfBytes, 0, 128);
                            if constexpr (PAIR)
                                ptx::tmem_cp_128x128b_pair(sf_tmem + h * kMetaTmemStride, d);
                            else
                                ptx::tmem_cp_128x128b(sf_tmem + h * kMetaTmemStride, d);
                        }
                    }
                    if constexpr (PAIR)
                        ptx::mma_commit_pair(sfr_bar(stage), static_cast<uint16_t>(1u << crank));
                    else
                        ptx::mma_commit_cta1(sfr_bar(stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if constexpr (T::kMX) {
                        if (pos == kScGroup - 1 || i == kb1 - kb0 - 1) {
                            // The slot's last copies issued: free it (in both CTAs of a pair, each
                            // of which refills its own) once they complete.
                            if constexpr (PAIR)
                                ptx::mma_commit_pair(sce_bar(sc_slot), 0x3);
                            else
                                ptx::mma_commit_cta1(sce_bar(sc_slot));
                            if (++sc_slot == kScSlots) {
                                sc_slot = 0;
                                sc_phase ^= 1u;
                            }
                        }
                    }
                }
            }
            // Every copy issued here completes before the TMEM is released.
            if constexpr (PAIR)
                ptx::mma_commit_pair(sdrain_bar, static_cast<uint16_t>(1u << crank));
            else
                ptx::mma_commit_cta1(sdrain_bar);
            wd.drain(sdrain_bar, 0);
        }
        __syncwarp();
    } else {
        // -------------------------------------------------------------------- epilogue
        const int ew = warp - kEpiWarp0;            // 0..3: staging buffers
        const int quad = warp & 3;                  // TMEM lane quadrant this warp may read
        const int row_in_cta = quad * 32 + lane;    // accumulator row of this thread
        const uint32_t stg0 = base + L::kStgOff + ew * L::kStgBufs * kStgBytes;
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        int acc = 0;
        uint32_t acc_phase = 0;
        int sbuf = 0;
        WorkIter it(p, unit, units);
        int64_t tile;
        int kb0, kb1;
        auto release_acc = [&]() {
            // Whole accumulator read: hand the buffer back to the MMA thread.
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR)
                    ptx::mbar_arrive_cluster(ptx::mapa_shared(acce_bar(acc), 0u));
                else
                    ptx::mbar_arrive(acce_bar(acc));
            }
        };
        while (it.next(p, tile, kb0, kb1)) {
            int64_t tm, tn;
            tile_coord(tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
            const bool ok = wd.wait(accf_bar(acc), acc_phase, kRoleEpilogue, tile, -1);
            if (!epilogue_bar_and(ok)) break;  // all four epilogue warps leave together
            ptx::tc_fence_after_sync();
            const int32_t y = static_cast<int32_t>(tm * kTileM + rank * kBM + quad * 32);
            const uint32_t tacc = tmem_base + lane_off + static_cast<uint32_t>(acc * BN);
            if (kAccBufs == 1 && kb0 == 0 && kb1 == p.num_kb) {
                // Whole tile, single accumulator: read the whole row of the accumulator into
                // registers (scaled, rounded to 16 bits) and hand the accumulator back before
                // storing, so that the next item's MMAs run while this tile is written.
                uint32_t h[BN / kEpiCols][32];
#pragma unroll
                for (int c = 0; c < BN / kEpiCols; ++c) {
                    uint32_t v[64];
                    uint32_t(&v0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
                    uint32_t(&v1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
                    ptx::tmem_ld_32x32b_x32(tacc + c * kEpiCols, v0);
                    ptx::tmem_ld_32x32b_x32(tacc + c * kEpiCols + 32, v1);
                    ptx::tmem_wait_ld();
                    scale_box<OUT_BF16>(v, static_cast<int32_t>(tn * BN + c * kEpiCols), y, lane, p);
                    pack_box<OUT_BF16>(v, h[c]);
                }
                release_acc();
#pragma unroll
                for (int c = 0; c < BN / kEpiCols; ++c) {
                    const int32_t x = static_cast<int32_t>(tn * BN + c * kEpiCols);
                    if (store_packed<L::kStgBufs>(h[c], x, y, lane, stg0 + sbuf * kStgBytes, &tmC, p))
                        sbuf ^= L::kStgBufs - 1;
                }
            } else if (kb0 == 0 && kb1 == p.num_kb) {
                // Whole tile: convert and store.
#pragma unroll 1
                for (int c = 0; c < BN / kEpiCols; ++c) {
                    uint32_t v[64];
                    uint32_t(&v0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
                    uint32_t(&v1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
                    ptx::tmem_ld_32x32b_x32(tacc + c * kEpiCols, v0);
                    ptx::tmem_ld_32x32b_x32(tacc + c * kEpiCols + 32, v1);
                    ptx::tmem_wait_ld();
                    if (c == BN / kEpiCols - 1) release_acc();
                    const int32_t x = static_cast<int32_t>(tn * BN + c * kEpiCols);
                    if (store_box<OUT_BF16, L::kStgBufs>(v, x, y, lane, stg0 + sbuf * kStgBytes, &tmC, p)) sbuf ^= L::kStgBufs - 1;
                }
            } else {
                // Part of a stream-K tile: park the fp32 partial sums in this unit's slot.
                // A slot holds float4 column groups group-major, rows inner, so each warp
                // store / load moves 512 contiguous bytes (32 rows of one column group).
                const int64_t tr = tile - p.dp_tiles;
                constexpr size_t kSlotF4 = static_cast<size_t>(kBM) * BN / 4;
                auto slot_f4 = [&](int64_t slot) {
                    return reinterpret_cast<float4*>(p.ws) + (static_cast<size_t>(slot) * CLUSTER + crank) * kSlotF4 +
                           row_in_cta;
                };
                int64_t first_unit, parts;
                sk_parts(p, tr, first_unit, parts);
                const int64_t my_part = unit - first_unit;
                int32_t* counter = p.counters + tr * CLUSTER + crank;
                // Sum all parts in K order (so the result does not depend on who arrives
                // last) and store.  With own_in_tmem this part's sums are read from TMEM at
                // its place in the order instead of from the workspace.
                auto reduce_and_store = [&](bool own_in_tmem) {
#pragma unroll 1
                    for (int c = 0; c < BN / kEpiCols; ++c) {
                        float s[64];
#pragma unroll
                        for (int i = 0; i < 64; ++i) s[i] = 0.0f;
#pragma unroll 2
                        for (int64_t part = 0; part < parts; ++part) {
                            if (own_in_tmem && part == my_part) {
                                uint32_t v[64];
                                uint32_t(&v0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
                                uint32_t(&v1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
                                ptx::tmem_ld_32x32b_x32(tacc + c * kEpiCols, v0);
                                ptx::tmem_ld_32x32b_x32(tacc + c * kEpiCols + 32, v1);
                                ptx::tmem_wait_ld();
#pragma unroll
                                for (int i = 0; i < 64; ++i) s[i] += __uint_as_float(v[i]);
                            } else {
                                const float4* s4 = slot_f4(sk_slot(p, first_unit + part, tr)) + c * 16 * kBM;
                                float4 f[16];
#pragma unroll
                                for (int q = 0; q < 16; ++q) f[q] = __ldcg(s4 + q * kBM);
#pragma unroll
                                for (int q = 0; q < 16; ++q) {
                                    s[4 * q] += f[q].x;
                                    s[4 * q + 1] += f[q].y;
                                    s[4 * q + 2] += f[q].z;
                                    s[4 * q + 3] += f[q].w;
                                }
                            }
                        }
                        if (own_in_tmem && c == BN / kEpiCols - 1) release_acc();
                        uint32_t v[64];
#pragma unroll
                        for (int i = 0; i < 64; ++i) v[i] = __float_as_uint(s[i]);
                        const int32_t x = static_cast<int32_t>(tn * BN + c * kEpiCols);
                        if (store_box<OUT_BF16, L::kStgBufs>(v, x, y, lane, stg0 + sbuf * kStgBytes, &tmC, p)) sbuf ^= L::kStgBufs - 1;
                    }
                };
                // Are all the other parts in already?  Then this part is the last: it skips
                // parking its own sums.  (Each other part parked its sums before counting
                // itself in, so what the count shows is visible.)
                if (ew == 0 && lane == 0) {
                    const bool last = atomicAdd(counter, 0) == parts - 1;
                    if (last) {
                        *counter = 0;  // every other part has counted itself in: ready for reuse
                        __threadfence();
                    }
                    *last_flag = last ? 1 : 0;
                }
                epilogue_bar_sync();
                if (*last_flag) {
                    reduce_and_store(true);
                } else {
                    float4* mine = slot_f4(sk_slot(p, unit, tr));
#pragma unroll 1
                    for (int c = 0; c < BN / kEpiCols; ++c) {
                        uint32_t v[64];
                        uint32_t(&v0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
                        uint32_t(&v1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
                        ptx::tmem_ld_32x32b_x32(tacc + c * kEpiCols, v0);
                        ptx::tmem_ld_32x32b_x32(tacc + c * kEpiCols + 32, v1);
                        ptx::tmem_wait_ld();
                        if (c == BN / kEpiCols - 1) release_acc();
#pragma unroll
                        for (int q = 0; q < 16; ++q)
                            mine[(c * 16 + q) * kBM] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                                                   __uint_as_float(v[4 * q + 2]),
                                                                   __uint_as_float(v[4 * q + 3]));
                    }
                    // Count this part in; if it turns out to be the last, sum every part.
                    __threadfence();
                    epilogue_bar_sync();
                    if (ew == 0 && lane == 0) {
                        const bool last = atomicAdd(counter, 1) == parts - 1;
                        if (last) {
                            *counter = 0;
                            __threadfence();
                        }
                        *last_flag = last ? 1 : 0;
                    }
                    epilogue_bar_sync();
                    if (*last_flag) reduce_and_store(false);
                }
            }
            if (++acc == kAccBufs) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0) ptx::bulk_wait_group_all();
        __syncwarp();
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if constexpr (PAIR) ptx::cluster_sync();  // neither CTA exits or frees TMEM while the peer may use it
    if (warp == kMmaWarp) {
        ptx::tc_fence_after_sync();
        if constexpr (PAIR)
            ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
        else
            ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
}

// The K == 0 case: A·B is the empty sum, so C = beta * C (C = 0 when beta == 0, without
// reading C).  Grid-stride over the M x N elements, row-major or column-major storage.
template <bool BF16>
__global__ void scale_c_kernel(uint16_t* C, int64_t M, int64_t N, int64_t ldc, int32_t col_major, float beta)
{
    const int64_t total = M * N;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = i / N, n = i - m * N;
        uint16_t* c = col_major ? C + n * ldc + m : C + m * ldc + n;
        const float f = beta != 0.0f ? beta * load16<BF16>(c) : 0.0f;
        *c = cvt16<BF16>(__float_as_uint(f));
    }
}

}  // namespace dtg

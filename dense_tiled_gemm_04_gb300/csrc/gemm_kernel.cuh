// Persistent warp-specialised tcgen05 GEMM for sm_103a: C = A·B, fp16/bf16 in, fp32
// accumulate in tensor memory (TMEM), fp16/bf16 out.
//
// Structure (the four steps of "张量缩并：mma 语法" -- fill, load, multiply, store -- with
// the load and the multiply on different warps so they overlap, which the same page
// names as the next step after its one-warp kernel):
//
//   warp 0        TMA producer: per K block, waits for a free ring stage, arms its "full"
//                 barrier with the byte count and issues the A and B tile loads.  Reads
//                 outside the tensor are zero-filled by the TMA unit ("NineToothed GEMM
//                 语法入门" §5: out-of-range reads contribute 0).
//   warp 1        MMA issuer (one thread): per K block, BK/16 tcgen05.mma into the TMEM
//                 accumulator, then tcgen05.commit releases the stage; after the tile's
//                 last K block a commit marks the accumulator full.  The first MMA of a
//                 tile overwrites (the zero-filled accumulator of §2), later ones add.
//   warps 2..5    epilogue: tcgen05.ld of the accumulator (each warp owns the 32 TMEM lanes
//                 of its lane quadrant), fp32 -> fp16/bf16 round-to-nearest-even, staging
//                 in 128-byte-swizzled shared memory and a TMA store that drops elements
//                 outside M x N (§5: masked write-back).
//
// The accumulator is double-buffered in TMEM (2 x BN fp32 columns), so the epilogue of
// tile t overlaps the main loop of tile t+1.  Tiles are walked persistently: CTA b takes
// tiles b, b + gridDim.x, ... in a grouped raster order (tile_coord).
//
// Every mbarrier wait is bounded (a watchdog on %globaltimer): on expiry the waiting
// thread records the place in the device error word, raises a CTA-wide abort flag, and
// all roles leave their loops; the producer then waits (bounded) for its in-flight
// loads, the MMA thread for its in-flight MMAs, the epilogue for its stores, and the
// TMEM is freed before the CTA exits.  No trap, no unbounded spin.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "sm103_ptx.cuh"

namespace dtg {

constexpr int kBM = 128;          // rows per tile (= MMA M, one TMEM lane per row)
constexpr int kBK = 64;           // K per ring stage: 64 x 2 B = one 128-byte swizzle row
constexpr int kUmmaK = 16;        // K per tcgen05.mma of kind::f16
constexpr int kThreads = 192;     // 6 warps
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kEpiWarp0 = 2;
constexpr int kEpiWarps = 4;
constexpr int kEpiCols = 64;                        // columns per staged TMA store box
constexpr int kStgBytes = 32 * kEpiCols * 2;        // one warp's 32 x 64 box, 4 KB

constexpr uint32_t kWaitSleepNs = 20000;           // longest single suspension of a waiting thread

// Error-word roles.
constexpr int kRoleProducer = 0, kRoleMma = 1, kRoleEpilogue = 2, kRoleDrain = 3;

struct KernelParams {
    int32_t M, N, K;
    int32_t tiles_m, tiles_n, num_kb, num_tiles;
    int32_t group_m;             // raster group (tile rows)
    int32_t fault_inject;        // test hook, see GEMM_OPT_FAULT_INJECT
    uint64_t timeout_ns;         // watchdog per wait
    int32_t* err;                // device error word [4]
    void* C;                     // output base, for the ragged-N edge written without TMA
    int64_t ldc;                 // output row pitch (elements)
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

template <int BN, int STAGES>
struct Smem {
    static constexpr int kABytes = kBM * kBK * 2;
    static constexpr int kBBytes = BN * kBK * 2;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kRing = STAGES * kStageBytes;
    static constexpr int kStgOff = kRing;
    static constexpr int kStg = kEpiWarps * 2 * kStgBytes;
    static constexpr int kBarOff = kStgOff + kStg;
    static constexpr int kNumBars = 2 * STAGES + 5;  // full, empty, acc_full[2], acc_empty[2], drain
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kTotal = kMiscOff + 16;     // tmem slot, abort flag
    static constexpr int kAlloc = kTotal + 1024;     // slack for aligning the base to 1 KB
    static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0, "swizzle atoms need 1 KB alignment");
    static constexpr int kTmemCols = 2 * BN;         // two accumulator buffers
    static_assert(kTmemCols == 32 || kTmemCols == 64 || kTmemCols == 128 || kTmemCols == 256 ||
                      kTmemCols == 512,
                  "TMEM allocations are powers of two");
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

// Instruction descriptor of tcgen05.mma.kind::f16: D fp32, A/B fp16 or bf16, A K-major,
// B K-major (TN) or N-major (NN), M x N shape.
template <bool BF16, bool B_MN_MAJOR, int M, int N>
__host__ __device__ constexpr uint32_t idesc_f16()
{
    return (1u << 4)                                  // D format: f32
           | ((BF16 ? 1u : 0u) << 7)                  // A format: 0 f16, 1 bf16
           | ((BF16 ? 1u : 0u) << 10)                 // B format
           | ((B_MN_MAJOR ? 1u : 0u) << 16)           // B major-ness
           | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

struct Watchdog {
    volatile int32_t* abort_flag;  // shared memory
    const KernelParams* p;
    uint32_t peer_abort = 0;       // shared::cluster address of the peer CTA's flag (CTA pairs), or 0

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

// Write the 32-row x 64-column box of C at (row y, column x) that this warp holds (lane =
// row, v = the 64 fp32 accumulator bit patterns of that row).  Normally the box goes
// through a 128-byte-swizzled staging buffer and one TMA store, which drops rows >= M and
// columns >= N (the masked write-back of "NineToothed GEMM 语法入门" §5).  A TMA store clips the inner dimension only
// to 16-byte granules, so when N is not a multiple of 8 the box that straddles column N
// is written with plain masked stores instead.  Returns true if the staging buffer was
// used (the caller then alternates buffers).
template <bool BF16>
__device__ __forceinline__ bool store_box(const uint32_t (&v)[64], int32_t x, int32_t y, int lane,
                                          uint32_t stg, const CUtensorMap* tmC, const KernelParams& p)
{
    if ((p.N & 7) != 0 && x + kEpiCols > p.N) {
        const int64_t row = static_cast<int64_t>(y) + lane;
        if (row < p.M && x < p.N) {
            uint16_t* crow = static_cast<uint16_t*>(p.C) + row * p.ldc;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                const int32_t col = x + ch * 8;
                if (col + 8 <= p.N) {  // a whole 16-byte chunk: one vector store
                    uint4 q;
                    q.x = pack2<BF16>(v[8 * ch + 0], v[8 * ch + 1]);
                    q.y = pack2<BF16>(v[8 * ch + 2], v[8 * ch + 3]);
                    q.z = pack2<BF16>(v[8 * ch + 4], v[8 * ch + 5]);
                    q.w = pack2<BF16>(v[8 * ch + 6], v[8 * ch + 7]);
                    *reinterpret_cast<uint4*>(crow + col) = q;
                } else {
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        const uint32_t two = pack2<BF16>(v[8 * ch + e], v[8 * ch + e + 1]);
                        if (col + e < p.N) crow[col + e] = static_cast<uint16_t>(two & 0xFFFFu);
                        if (col + e + 1 < p.N) crow[col + e + 1] = static_cast<uint16_t>(two >> 16);
                    }
                }
            }
        }
        return false;
    }
    // The staging buffer is reusable once the store issued from it two boxes ago has
    // finished reading it.
    if (lane == 0) ptx::bulk_wait_group_read<1>();
    __syncwarp();
    const uint32_t row = stg + lane * 128;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        // 16-byte chunk ch of this row lands at chunk (ch ^ row%8): the 128-byte swizzle
        // the TMA store expects.
        const uint32_t addr = row + ((ch ^ (lane & 7)) << 4);
        ptx::st_shared_v4(addr, pack2<BF16>(v[8 * ch + 0], v[8 * ch + 1]), pack2<BF16>(v[8 * ch + 2], v[8 * ch + 3]),
                          pack2<BF16>(v[8 * ch + 4], v[8 * ch + 5]), pack2<BF16>(v[8 * ch + 6], v[8 * ch + 7]));
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (x < p.N && y < p.M) ptx::tma_store_2d(tmC, stg, x, y);
        ptx::bulk_commit_group();
    }
    return true;
}

template <int BN, int STAGES, bool BF16, bool B_MN_MAJOR>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const KernelParams p)
{
    using L = Smem<BN, STAGES>;
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
    uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    volatile int32_t* const abort_flag = reinterpret_cast<volatile int32_t*>(smem + L::kMiscOff + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(accf_bar(b), 1);
            ptx::mbar_init(acce_bar(b), kEpiWarps);
        }
        ptx::mbar_init(drain_bar, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
        ptx::prefetch_tmap(&tmC);
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), L::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    const Watchdog wd{abort_flag, &p};
    const int num_kb = p.num_kb;

    if (warp == kProducerWarp) {
        if (lane == 0) {
            // ---------------------------------------------------------------- producer
            uint32_t armed_mask = 0, armed_parity = 0;  // per stage: armed at least once, last parity
            int stage = 0;
            uint32_t phase = 0;
            bool injected = false;
            for (int64_t t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
                int64_t tm, tn;
                tile_coord(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
                const int32_t y_a = static_cast<int32_t>(tm * kBM);
                const int32_t n0 = static_cast<int32_t>(tn * BN);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!wd.wait(empty_bar(stage), phase ^ 1u, kRoleProducer, t, kb)) goto producer_done;
                    if (p.fault_inject && !injected && blockIdx.x == 0 && kb == (num_kb > 1 ? 1 : 0)) {
                        injected = true;  // leave this stage unarmed: its consumer must time out
                    } else {
                        const uint32_t sa = base + stage * L::kStageBytes;
                        const uint32_t sb = sa + L::kABytes;
                        const int32_t k0 = kb * kBK;
                        ptx::mbar_arrive_expect_tx(full_bar(stage), L::kStageBytes);
                        ptx::tma_load_2d(sa, &tmA, k0, y_a, full_bar(stage));
                        if constexpr (B_MN_MAJOR) {
                            // B stored K x N: BN/64 boxes of 64 (N) x 64 (K), each 8 KB.
#pragma unroll
                            for (int q = 0; q < BN / 64; ++q)
                                ptx::tma_load_2d(sb + q * (64 * kBK * 2), &tmB, n0 + q * 64, k0, full_bar(stage));
                        } else {
                            // B stored N x K: one box of 64 (K) x BN (N rows).
                            ptx::tma_load_2d(sb, &tmB, k0, n0, full_bar(stage));
                        }
                        armed_mask |= 1u << stage;
                        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Tail: wait (bounded) until the MMA thread has released every stage this
            // producer filled, so no tcgen05.commit arrival is still heading for this
            // CTA's barriers when it leaves.
            for (int i = 0; i < STAGES; ++i) {
                if (!wd.wait(empty_bar(stage), phase ^ 1u, kRoleProducer, -1, i)) break;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        producer_done:
            // Wait (bounded) for every load this thread issued, so none is in flight at exit.
            for (int s = 0; s < STAGES; ++s)
                if (armed_mask & (1u << s)) wd.drain(full_bar(s), (armed_parity >> s) & 1u);
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            // ---------------------------------------------------------------- MMA issuer
            constexpr uint32_t idesc = idesc_f16<BF16, B_MN_MAJOR, kBM, BN>();
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool aborted = false;
            if (num_kb > 0) {
                for (int64_t t = blockIdx.x; t < p.num_tiles && !aborted; t += gridDim.x) {
                    if (!wd.wait(acce_bar(acc), acc_phase ^ 1u, kRoleMma, t, -1)) {
                        aborted = true;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                    for (int kb = 0; kb < num_kb; ++kb) {
                        if (!wd.wait(full_bar(stage), phase, kRoleMma, t, kb)) {
                            aborted = true;
                            break;
                        }
                        ptx::tc_fence_after_sync();
                        const uint32_t sa = base + stage * L::kStageBytes;
                        const uint32_t sb = sa + L::kABytes;
#pragma unroll
                        for (int k = 0; k < kBK / kUmmaK; ++k) {
                            // A (K-major, 128B swizzle): the k-th 16-column slice starts 32 B
                            // further along each 128-byte row; 8-row groups are 1 KB apart.
                            const uint64_t adesc = smem_desc_sw128(sa + k * 32, 16, 1024);
                            uint64_t bdesc;
                            if constexpr (B_MN_MAJOR) {
                                // B (N-major): rows are K; the k-th slice is 16 rows (2 KB) on;
                                // 64-wide N blocks are 8 KB apart (LBO), 8-row K groups 1 KB (SBO).
                                bdesc = smem_desc_sw128(sb + k * 2048, 64 * kBK * 2, 1024);
                            } else {
                                bdesc = smem_desc_sw128(sb + k * 32, 16, 1024);
                            }
                            ptx::mma_f16_cta1(d_tmem, adesc, bdesc, idesc, (kb | k) != 0 ? 1u : 0u);
                        }
                        ptx::mma_commit_cta1(empty_bar(stage));  // stage free once these MMAs finish
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (aborted) break;
                    ptx::mma_commit_cta1(accf_bar(acc));  // accumulator complete
                    if (++acc == 2) {
                        acc = 0;
                        acc_phase ^= 1u;
                    }
                }
            }
            if (aborted) {
                // Let every MMA issued so far finish before the TMEM is released.
                ptx::mma_commit_cta1(drain_bar);
                wd.drain(drain_bar, 0);
            }
        }
        __syncwarp();
    } else {
        // -------------------------------------------------------------------- epilogue
        const int ew = warp - kEpiWarp0;            // 0..3: staging buffers
        const int quad = warp & 3;                  // TMEM lane quadrant this warp may read
        const uint32_t stg0 = base + L::kStgOff + ew * 2 * kStgBytes;
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        int acc = 0;
        uint32_t acc_phase = 0;
        int sbuf = 0;
        for (int64_t t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
            int64_t tm, tn;
            tile_coord(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
            if (num_kb > 0) {
                const bool ok = wd.wait(accf_bar(acc), acc_phase, kRoleEpilogue, t, -1);
                if (!__all_sync(0xffffffffu, ok)) break;
                ptx::tc_fence_after_sync();
            }
            const int32_t y = static_cast<int32_t>(tm * kBM + quad * 32);
#pragma unroll 1
            for (int c = 0; c < BN / kEpiCols; ++c) {
                uint32_t v[64];
                if (num_kb > 0) {
                    const uint32_t ta = tmem_base + lane_off + static_cast<uint32_t>(acc * BN + c * kEpiCols);
                    uint32_t (&v0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
                    uint32_t (&v1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
                    ptx::tmem_ld_32x32b_x32(ta, v0);
                    ptx::tmem_ld_32x32b_x32(ta + 32, v1);
                    ptx::tmem_wait_ld();
                    if (c == BN / kEpiCols - 1) {
                        // Whole accumulator read: hand the buffer back to the MMA warp.
                        ptx::tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(acce_bar(acc));
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 64; ++i) v[i] = 0u;  // K == 0: the empty sum
                }
                const int32_t x = static_cast<int32_t>(tn * BN + c * kEpiCols);
                if (store_box<BF16>(v, x, y, lane, stg0 + sbuf * kStgBytes, &tmC, p)) sbuf ^= 1;
            }
            if (num_kb > 0 && ++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0) ptx::bulk_wait_group_all();
        __syncwarp();
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem_base, L::kTmemCols);
    }
}

// C[M x N] = 0 for the K == 0 case (the empty sum).  Grid-stride over rows and columns.
template <typename T>
__global__ void zero_fill_kernel(T* C, int64_t M, int64_t N, int64_t ldc)
{
    const int64_t total = M * N;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = i / N, n = i - m * N;
        C[m * ldc + n] = T(0.0f);
    }
}

}  // namespace dtg

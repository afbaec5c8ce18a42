// Two-CTA (CTA pair) variant of the persistent tcgen05 GEMM: a cluster of two CTAs on two
// SMs computes one 256 x 256 output tile with tcgen05.mma.cta_group::2 (M = 256, N = 256).
//
// The idea is the two-warpgroup kernel of "张量缩并：mma 语法" (two workers share one B tile
// while each takes its own rows of A), moved to the SM level: CTA r of the pair loads rows
// [128 r, 128 r + 128) of the A tile and columns [128 r, 128 r + 128) of the B tile into its
// own shared memory; one thread of the leader CTA (rank 0) issues the pair MMA, which reads
// A and B halves from both CTAs and writes each CTA's 128 accumulator rows into that CTA's
// tensor memory.  Per SM this halves the shared-memory bytes of B per MMA compared with a
// 128 x 256 tile on one SM.
//
// Synchronisation across the pair:
//   full[s]      lives in the leader.  The leader's producer arms it with the bytes of both
//                CTAs; both producers' TMA loads complete on it (.cta_group::2 loads may
//                signal the peer's barrier).
//   empty[s]     in both CTAs; the leader's MMA commit arrives on both (multicast).
//   acc_full[b]  in both CTAs; the leader's commit after a tile's last K block, multicast.
//   acc_empty[b] lives in the leader, count 8: the 4 epilogue warps of each CTA arrive after
//                reading their accumulator rows.
// Every wait is bounded as in the one-CTA kernel; a failure also raises the peer's abort
// flag, and both CTAs meet at a cluster barrier before the pair's TMEM is freed and either
// CTA exits (no CTA leaves while its peer may still touch its shared memory).
#pragma once
#include "gemm_kernel.cuh"

namespace dtg {

constexpr int kPairBM = 256;     // rows per pair tile (128 per CTA)
constexpr int kPairBN = 256;     // columns per pair tile (B: 128 rows/columns per CTA)
constexpr int kPairTmemCols = 512;

template <int STAGES>
using PairSmem = Smem<128, STAGES>;  // per CTA: A 128 x 64 and B half 128 x 64 per stage

template <int STAGES, bool BF16, bool B_MN_MAJOR>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_tcgen05_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmC, const KernelParams p)
{
    using L = PairSmem<STAGES>;
    extern __shared__ uint8_t smem_raw[];
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
    const uint32_t rank = ptx::cluster_ctarank();  // 0 = leader, 1 = peer
    const bool leader = rank == 0;
    const int64_t cluster = ptx::cluster_id_x();
    const int64_t clusters = ptx::num_clusters_x();

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(accf_bar(b), 1);
            ptx::mbar_init(acce_bar(b), 2 * kEpiWarps);
        }
        ptx::mbar_init(drain_bar, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
        ptx::prefetch_tmap(&tmC);
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc_pair(ptx::smem_addr(tmem_slot), kPairTmemCols);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before_sync();
    ptx::cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    Watchdog wd{abort_flag, &p};
    wd.peer_abort = ptx::mapa_shared(ptx::smem_addr(const_cast<int32_t*>(abort_flag)), rank ^ 1u);
    const int num_kb = p.num_kb;

    if (warp == kProducerWarp) {
        if (lane == 0) {
            // ---------------------------------------------------------------- producer (both CTAs)
            uint32_t armed_mask = 0, armed_parity = 0;  // leader only: stages armed, last parity
            int stage = 0;
            uint32_t phase = 0;
            bool injected = false;
            for (int64_t t = cluster; t < p.num_tiles; t += clusters) {
                int64_t tm, tn;
                tile_coord(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
                const int32_t y_a = static_cast<int32_t>(tm * kPairBM + rank * 128);
                const int32_t n_b = static_cast<int32_t>(tn * kPairBN + rank * 128);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!wd.wait(empty_bar(stage), phase ^ 1u, kRoleProducer, t, kb)) goto producer_done;
                    const bool skip = p.fault_inject && !injected && leader && cluster == 0 &&
                                      kb == (num_kb > 1 ? 1 : 0);
                    if (skip) {
                        injected = true;  // leave this stage unarmed: the MMA wait must time out
                    } else {
                        const uint32_t sa = base + stage * L::kStageBytes;
                        const uint32_t sb = sa + L::kABytes;
                        const int32_t k0 = kb * kBK;
                        const uint32_t fb = ptx::mapa_shared(full_bar(stage), 0);  // the leader's barrier
                        if (leader) {
                            ptx::mbar_arrive_expect_tx(full_bar(stage), 2u * L::kStageBytes);
                            armed_mask |= 1u << stage;
                            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                        }
                        ptx::tma_load_2d_pair(sa, &tmA, k0, y_a, fb);
                        if constexpr (B_MN_MAJOR) {
                            // B stored K x N: this CTA's 128 columns as two 64 (N) x 64 (K) boxes.
                            ptx::tma_load_2d_pair(sb, &tmB, n_b, k0, fb);
                            ptx::tma_load_2d_pair(sb + 64 * kBK * 2, &tmB, n_b + 64, k0, fb);
                        } else {
                            // B stored N x K: this CTA's 128 rows of N, 64 of K.
                            ptx::tma_load_2d_pair(sb, &tmB, k0, n_b, fb);
                        }
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
            // The leader's full barriers count both CTAs' loads: waiting on them (bounded)
            // covers every load in flight for the pair.
            if (leader)
                for (int s = 0; s < STAGES; ++s)
                    if (armed_mask & (1u << s)) wd.drain(full_bar(s), (armed_parity >> s) & 1u);
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0 && leader) {
            // ---------------------------------------------------------------- MMA issuer (leader)
            constexpr uint32_t idesc = idesc_f16<BF16, B_MN_MAJOR, kPairBM, kPairBN>();
            constexpr uint16_t kBoth = 0x3;
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool aborted = false;
            if (num_kb > 0) {
                for (int64_t t = cluster; t < p.num_tiles && !aborted; t += clusters) {
                    if (!wd.wait(acce_bar(acc), acc_phase ^ 1u, kRoleMma, t, -1)) {
                        aborted = true;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kPairBN);
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
                            const uint64_t adesc = smem_desc_sw128(sa + k * 32, 16, 1024);
                            uint64_t bdesc;
                            if constexpr (B_MN_MAJOR)
                                bdesc = smem_desc_sw128(sb + k * 2048, 64 * kBK * 2, 1024);
                            else
                                bdesc = smem_desc_sw128(sb + k * 32, 16, 1024);
                            ptx::mma_f16_pair(d_tmem, adesc, bdesc, idesc, (kb | k) != 0 ? 1u : 0u);
                        }
                        ptx::mma_commit_pair_mc(empty_bar(stage), kBoth);  // frees the stage in both CTAs
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (aborted) break;
                    ptx::mma_commit_pair_mc(accf_bar(acc), kBoth);  // both CTAs' accumulators complete
                    if (++acc == 2) {
                        acc = 0;
                        acc_phase ^= 1u;
                    }
                }
            }
            if (aborted) {
                ptx::mma_commit_pair_mc(drain_bar, 0x1);
                wd.drain(drain_bar, 0);
            }
        }
        __syncwarp();
    } else {
        // -------------------------------------------------------------------- epilogue (both CTAs)
        const int ew = warp - kEpiWarp0;
        const int quad = warp & 3;
        const uint32_t stg0 = base + L::kStgOff + ew * 2 * kStgBytes;
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        int acc = 0;
        uint32_t acc_phase = 0;
        int sbuf = 0;
        for (int64_t t = cluster; t < p.num_tiles; t += clusters) {
            int64_t tm, tn;
            tile_coord(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
            if (num_kb > 0) {
                const bool ok = wd.wait(accf_bar(acc), acc_phase, kRoleEpilogue, t, -1);
                if (!__all_sync(0xffffffffu, ok)) break;
                ptx::tc_fence_after_sync();
            }
            const int32_t y = static_cast<int32_t>(tm * kPairBM + rank * 128 + quad * 32);
#pragma unroll 1
            for (int c = 0; c < kPairBN / kEpiCols; ++c) {
                uint32_t v[64];
                if (num_kb > 0) {
                    const uint32_t ta = tmem_base + lane_off + static_cast<uint32_t>(acc * kPairBN + c * kEpiCols);
                    uint32_t(&v0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
                    uint32_t(&v1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
                    ptx::tmem_ld_32x32b_x32(ta, v0);
                    ptx::tmem_ld_32x32b_x32(ta + 32, v1);
                    ptx::tmem_wait_ld();
                    if (c == kPairBN / kEpiCols - 1) {
                        // This CTA's rows are read: tell the leader's MMA thread.
                        ptx::tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(acce_bar(acc), 0));
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 64; ++i) v[i] = 0u;
                }
                const int32_t x = static_cast<int32_t>(tn * kPairBN + c * kEpiCols);
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
    ptx::cluster_sync();  // neither CTA exits or frees TMEM while the peer may still use it
    if (warp == kMmaWarp) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc_pair(tmem_base, kPairTmemCols);
    }
}

}  // namespace dtg

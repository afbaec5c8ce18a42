// The set of kernel instantiations the host can launch, and how it names them.
//
// Each operand type's instantiations live in a translation unit of their own
// (kernels_f16.cu, kernels_bf16.cu, kernels_e4m3.cu, kernels_e5m2.cu, kernels_mx.cu,
// kernels_sparse.cu) so that nvcc
// compiles them in parallel; the host reaches them through the choice_* functions below,
// which return the kernel's address and launch shape.
#pragma once

#include "gemm_kernel.cuh"

namespace dtg {

constexpr int kPairStages = 6;  // ring depth of the 256 x 256 CTA-pair kernels

// Which kernel instantiation a plan launches.
struct KernelChoice {
    int config;
    int bm, bn;     // output tile of one CTA (1-CTA) or of the pair
    int b_box;      // rows (TN) / columns (NN) of B one CTA loads per stage
    int stage_k;    // K elements per ring stage (one 128-byte row of B)
    int n_block;    // NN: N elements per B box (128 bytes)
    int a_stage_k;  // stored A elements per stage row (stage_k, or half of it for a 2:4-sparse A)
    int stages;
    int cluster;    // CTAs per cluster
    const void* fn;
    int smem;
    int threads = kThreads;  // per CTA (kThreadsSide for the block-scaled and sparse kernels)
};

template <int BN, int STAGES, int IN, bool OUT_BF16, bool NN>
KernelChoice one_cta_choice(int config)
{
    return {config, kBM, BN, BN, Operand<IN>::kStageK, Operand<IN>::kNBlock, Operand<IN>::kAStageK, STAGES, 1,
            reinterpret_cast<const void*>(&gemm_tcgen05_kernel<BN, STAGES, IN, OUT_BF16, NN, 1>),
            KernelLayout<BN, STAGES, IN, false>::S::kAlloc,
            (Operand<IN>::kMX || Operand<IN>::kSparse) ? kThreadsSide : kThreads};
}

template <int IN, bool OUT_BF16, bool NN>
KernelChoice choice_for(int config)
{
    if (config == 3)  // GEMM_CONFIG_256x256
        return {3, 2 * kBM, 256, 128, Operand<IN>::kStageK, Operand<IN>::kNBlock, Operand<IN>::kAStageK,
                kPairStages, 2,
                reinterpret_cast<const void*>(&gemm_tcgen05_kernel<256, kPairStages, IN, OUT_BF16, NN, 2>),
                KernelLayout<256, kPairStages, IN, true>::S::kAlloc};
    if constexpr (Operand<IN>::kBytes == 2) {
        if (config == 4)  // GEMM_CONFIG_128x64: 24 KB stages (16-bit operands: 8-bit ones take 128 x 128)
            return one_cta_choice<64, 8, IN, OUT_BF16, NN>(config);
    }
    if (config == 2 || config == 4)  // GEMM_CONFIG_128x128
        return one_cta_choice<128, 6, IN, OUT_BF16, NN>(2);
    return one_cta_choice<256, 4, IN, OUT_BF16, NN>(1);  // GEMM_CONFIG_128x256
}

template <int IN, bool OUT_BF16>
KernelChoice choice_for_layout(int config, bool nn)
{
    return nn ? choice_for<IN, OUT_BF16, true>(config) : choice_for<IN, OUT_BF16, false>(config);
}

// config: GEMM_CONFIG_128x256, _128x128, _128x64 or _256x256 (never AUTO).
KernelChoice choice_f16(int config, bool nn);
KernelChoice choice_bf16(int config, bool nn);
KernelChoice choice_e4m3(int config, bool out_bf16, bool nn);
KernelChoice choice_e5m2(int config, bool out_bf16, bool nn);
// Block-scaled 8-bit operands: config GEMM_CONFIG_256x256 (the CTA pair) or anything else (the
// one-CTA 128 x 256 tile).
KernelChoice choice_mx(int config, bool e5m2, bool out_bf16, bool nn);
// 2:4-sparse A, fp16 or bf16 (C of the same type): config GEMM_CONFIG_256x256 (the CTA pair) or
// anything else (the one-CTA 128 x 256 tile).
KernelChoice choice_sparse(int config, bool bf16, bool nn);

}  // namespace dtg

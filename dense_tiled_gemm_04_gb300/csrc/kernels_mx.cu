// Block-scaled E4M3 / E5M2 operands (one E8M0 scale per 32 K elements), fp16 or bf16 output:
// the one-CTA 128 x 256 tile and the 256 x 256 CTA pair.
#include "kernel_set.cuh"

namespace dtg {
namespace {
constexpr int kMxPairStages = 6;

template <int IN, bool OUT_BF16, bool NN>
KernelChoice mx_choice(int config)
{
    if (config == 3)  // GEMM_CONFIG_256x256
        return {config, 2 * kBM, 256, 128, Operand<IN>::kStageK, Operand<IN>::kNBlock, Operand<IN>::kAStageK,
                kMxPairStages, 2,
                reinterpret_cast<const void*>(&gemm_tcgen05_kernel<256, kMxPairStages, IN, OUT_BF16, NN, 2>),
                KernelLayout<256, kMxPairStages, IN, true>::S::kAlloc, kThreadsSide};
    return one_cta_choice<256, 4, IN, OUT_BF16, NN>(1);
}

template <int IN, bool OUT_BF16>
KernelChoice mx_layout(int config, bool nn)
{
    return nn ? mx_choice<IN, OUT_BF16, true>(config) : mx_choice<IN, OUT_BF16, false>(config);
}
}  // namespace

KernelChoice choice_mx(int config, bool e5m2, bool out_bf16, bool nn)
{
    if (e5m2) return out_bf16 ? mx_layout<5, true>(config, nn) : mx_layout<5, false>(config, nn);
    return out_bf16 ? mx_layout<4, true>(config, nn) : mx_layout<4, false>(config, nn);
}
}  // namespace dtg

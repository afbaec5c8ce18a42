// 2:4-sparse A (kind::f16 .sp), fp16 or bf16 operands and output: the one-CTA 128 x 256 tile
// and the 256 x 256 CTA pair.
#include "kernel_set.cuh"

namespace dtg {
namespace {
// A sparse stage is consumed in two MMAs (half the time of a dense one), so the ring needs
// more stages for the same lead over the loads: 7 of 28 KB per CTA, with one staging buffer.
constexpr int kSparsePairStages = 7;

template <int IN, bool BF16, bool NN>
KernelChoice sparse_choice(int config)
{
    if (config == 3)  // GEMM_CONFIG_256x256
        return {config, 2 * kBM, 256, 128, Operand<IN>::kStageK, Operand<IN>::kNBlock, Operand<IN>::kAStageK,
                kSparsePairStages, 2,
                reinterpret_cast<const void*>(&gemm_tcgen05_kernel<256, kSparsePairStages, IN, BF16, NN, 2>),
                KernelLayout<256, kSparsePairStages, IN, true>::S::kAlloc, kThreadsSide};
    return one_cta_choice<256, 4, IN, BF16, NN>(1);
}
}  // namespace

KernelChoice choice_sparse(int config, bool bf16, bool nn)
{
    if (bf16) return nn ? sparse_choice<7, true, true>(config) : sparse_choice<7, true, false>(config);
    return nn ? sparse_choice<6, false, true>(config) : sparse_choice<6, false, false>(config);
}
}  // namespace dtg

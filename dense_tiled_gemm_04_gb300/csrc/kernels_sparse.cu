// 2:4-sparse A (kind::f16 .sp), fp16 or bf16 operands and output.
#include "kernel_set.cuh"

namespace dtg {
namespace {
template <int IN, bool BF16>
KernelChoice sparse_choice(bool nn)
{
    return nn ? one_cta_choice<256, 4, IN, BF16, true>(1) : one_cta_choice<256, 4, IN, BF16, false>(1);
}
}  // namespace

KernelChoice choice_sparse(bool bf16, bool nn) { return bf16 ? sparse_choice<7, true>(nn) : sparse_choice<6, false>(nn); }
}  // namespace dtg

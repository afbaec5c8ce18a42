// Block-scaled E4M3 / E5M2 operands (one E8M0 scale per 32 K elements), fp16 or bf16 output.
#include "kernel_set.cuh"

namespace dtg {
namespace {
template <int IN, bool OUT_BF16>
KernelChoice mx_choice(bool nn)
{
    return nn ? one_cta_choice<256, 4, IN, OUT_BF16, true>(1) : one_cta_choice<256, 4, IN, OUT_BF16, false>(1);
}
}  // namespace

KernelChoice choice_mx(bool e5m2, bool out_bf16, bool nn)
{
    if (e5m2) return out_bf16 ? mx_choice<5, true>(nn) : mx_choice<5, false>(nn);
    return out_bf16 ? mx_choice<4, true>(nn) : mx_choice<4, false>(nn);
}
}  // namespace dtg

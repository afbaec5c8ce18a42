// E5M2 operands, fp16 or bf16 output.
#include "kernel_set.cuh"

namespace dtg {
KernelChoice choice_e5m2(int config, bool out_bf16, bool nn)
{
    return out_bf16 ? choice_for_layout<3, true>(config, nn) : choice_for_layout<3, false>(config, nn);
}
}  // namespace dtg

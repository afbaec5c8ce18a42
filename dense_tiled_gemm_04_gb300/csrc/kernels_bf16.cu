// bf16 operands, bf16 output.
#include "kernel_set.cuh"

namespace dtg {
KernelChoice choice_bf16(int config, bool nn) { return choice_for_layout<1, true>(config, nn); }
}  // namespace dtg

// fp16 operands, fp16 output.
#include "kernel_set.cuh"

namespace dtg {
KernelChoice choice_f16(int config, bool nn) { return choice_for_layout<0, false>(config, nn); }
}  // namespace dtg

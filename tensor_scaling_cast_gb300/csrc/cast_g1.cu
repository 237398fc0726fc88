// Grouped cast kernels for groups of up to 1 tensor per launch (see cast_kernels.cuh).
#include "cast_kernels.cuh"

namespace fp8q {
FP8Q_CAST_GROUP_INSTANCES(, 1)
}  // namespace fp8q

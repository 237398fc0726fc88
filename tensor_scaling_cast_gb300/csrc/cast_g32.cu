// Grouped cast kernels for groups of up to 32 tensors per launch (see cast_kernels.cuh).
#include "cast_kernels.cuh"

namespace fp8q {
FP8Q_CAST_GROUP_INSTANCES(, 32)
}  // namespace fp8q

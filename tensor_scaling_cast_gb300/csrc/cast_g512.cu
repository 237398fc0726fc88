// Grouped cast kernels for groups of up to 512 tensors per launch (see cast_kernels.cuh).
#include "cast_kernels.cuh"

namespace fp8q {
FP8Q_CAST_GROUP_INSTANCES(, 512)
}  // namespace fp8q

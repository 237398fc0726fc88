// Grouped-cast dispatch and the dynamic loss-scale update.  The kernels of
// the fused per-tensor cast live in cast_kernels.cuh, instantiated per group
// size in cast_g1.cu, cast_g32.cu and cast_g512.cu.
#include <cuda_runtime.h>

#include "cast_kernels.cuh"

namespace fp8q {

FP8Q_CAST_GROUP_INSTANCES(extern, 1)
FP8Q_CAST_GROUP_INSTANCES(extern, 32)
FP8Q_CAST_GROUP_INSTANCES(extern, kMaxGroup)

template <int KIND>
static cudaError_t launch_group(const GroupHeader& h, const TensorDesc* d, int count,
                                cudaStream_t s, int* launches) {
  if (count <= 1) return launch_group_t<1, KIND>(h, d, count, s, launches);
  if (count <= 32) return launch_group_t<32, KIND>(h, d, count, s, launches);
  return launch_group_t<kMaxGroup, KIND>(h, d, count, s, launches);
}

cudaError_t launch_cast_group(const GroupHeader& h, const TensorDesc* d, int count,
                              cudaStream_t s, int* launches) {
  return h.underflow ? launch_group<2>(h, d, count, s, launches) : launch_group<1>(h, d, count, s, launches);
}

cudaError_t launch_amax_group(const GroupHeader& h, const TensorDesc* d, int count,
                              cudaStream_t s, int* launches) {
  return launch_group<0>(h, d, count, s, launches);
}

// ---- dynamic loss scaling ----------------------------------------------------
//
// One CTA: "was any input of this step NaN or Inf?" over the per-tensor
// non-finite counts, then the state machine ("Mixed Precision FP16/BF16/FP8":
// on Inf/NaN halve the scale and skip the step; after growth_interval clean
// steps in a row double it), clamped to [min_scale, max_scale].
__global__ void loss_scale_update_kernel(LossScaleState* st, const unsigned long long* nonfinite,
                                         int count, float* scale_out, int* skip_out) {
  int found = 0;
  for (int i = threadIdx.x; i < count; i += blockDim.x) found |= nonfinite[i] != 0ull;
  found = __syncthreads_or(found);
  if (threadIdx.x != 0) return;
  if (found) {
    st->scale = fmaxf(st->min_scale, st->scale * 0.5f);
    st->good = 0;
  } else if (++st->good >= st->growth_interval) {
    st->scale = fminf(st->max_scale, st->scale * 2.0f);
    st->good = 0;
  }
  st->last_skip = found;
  st->updates = st->updates + 1;
  if (scale_out) *scale_out = st->scale;
  if (skip_out) *skip_out = found;
}

cudaError_t launch_loss_scale_update(LossScaleState* st, const unsigned long long* nonfinite, int count,
                                     float* scale_out, int* skip_out, cudaStream_t s, int* launches) {
  loss_scale_update_kernel<<<1, kThreads, 0, s>>>(st, nonfinite, count, scale_out, skip_out);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace fp8q

// Per-tensor scaling state on the device: the statistic a cast's exponent
// comes from, and the finish that the CTA completing a tensor performs.
// Shared by the grouped cast and the cast-transpose kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8q_device.cuh"
#include "fp8q_internal.cuh"

namespace fp8q {

// Window maximum of a tensor's history (called by one full warp).
static __device__ __forceinline__ uint32_t window_max(const DevState* st) {
  const int count = __ldcg(&st->count);
  uint32_t a = 0;
  for (int i = threadIdx.x & 31; i < count; i += 32) a = max(a, __ldcg(&st->ring[i]));
  return __reduce_max_sync(0xFFFFFFFFu, a);
}

// Exponent of this cast.  With a recompute interval k > 1 the previous
// exponent is kept unless the number of earlier casts is a multiple of k
// (phase = casts mod k, kept by the finishing CTA).
static __device__ __forceinline__ int state_exp(const DevState* st, uint32_t a_w) {
  const int prev = __ldcg(&st->prev_e);
  const bool has_prev = __ldcg(&st->has_prev) != 0;
  if (has_prev && __ldcg(&st->phase) != 0) return prev;
  return pick_exp(a_w, __ldcg(&st->format), __ldcg(&st->margin), __ldcg(&st->hyst), prev, has_prev);
}

// Statistic of the smoothed estimator: the running average, or NaN (keep
// the previous exponent) while no finite amax has been seen.
static __device__ __forceinline__ uint32_t smoothed_stat(const DevState* st) {
  return __ldcg(&st->has_avg) ? (__float_as_uint(__ldcg(&st->avg)) & 0x7FFFFFFFu) : 0x7FC00000u;
}

// Warp 0: the statistic of this cast (window maximum, running average or
// current-scaling pre-pass amax) and the exponent, published in *s_e.
static __device__ __forceinline__ void warp_exp(const DevState* st, int mode, int* s_e) {
  uint32_t a_w;
  if (mode == kDelayed)
    a_w = (__ldcg(&st->estimator) == FP8Q_EST_SMOOTHED) ? smoothed_stat(st) : window_max(st);
  else
    a_w = __ldcg(&st->pre_amax);
  if (threadIdx.x == 0) *s_e = state_exp(st, a_w);
}

// Publish one cast's results (amax a, clipped, non-finite and underflow
// counts, exponent e) and advance the handle's state.  Thread 0 of the CTA
// that completes the tensor.
static __device__ void publish_and_advance(DevState* st, const GroupHeader& h, int t, int e, uint32_t a,
                                           unsigned long long cl, unsigned long long nf,
                                           unsigned long long uf) {
  if (a > 0x7F800000u) a = 0x7FC00000u;        // canonical NaN
  const int idx = h.out_offset + t;
  if (h.amax) h.amax[idx] = __uint_as_float(a);
  if (h.scale_inv) h.scale_inv[idx] = pow2f(-e);
  if (h.clipped) h.clipped[idx] = cl;
  if (h.nonfinite) h.nonfinite[idx] = nf;
  if (h.underflow) h.underflow[idx] = uf;
  const int W = st->window;
  if (W > 0) {
    const int hd = st->head;
    st->ring[hd] = a;
    st->head = (hd + 1 == W) ? 0 : hd + 1;
    if (st->count < W) st->count = st->count + 1;
  }
  if (st->estimator == FP8Q_EST_SMOOTHED && a < 0x7F800000u) {
    // avg <- avg + alpha * (amax - avg): three fp32 roundings, no FMA
    const float af = __uint_as_float(a);
    st->avg = st->has_avg ? __fadd_rn(st->avg, __fmul_rn(st->alpha, __fsub_rn(af, st->avg))) : af;
    st->has_avg = 1;
  }
  st->prev_e = e;
  st->has_prev = 1;
  st->steps = st->steps + 1;
  st->phase = (st->phase + 1 >= st->interval) ? 0 : st->phase + 1;
  st->amax_acc = 0u;
  st->clip_acc = 0ull;
  st->nonfinite_acc = 0ull;
  st->underflow_acc = 0ull;
  st->pre_amax = 0u;
  st->ticket = 0u;
}

// Thread 0 of the CTA whose ticket completes the tensor: the totals are the
// accumulators every CTA of the tensor added into.
static __device__ void finish_tensor(DevState* st, const GroupHeader& h, int t, int e) {
  __threadfence();
  const uint32_t a = atomicAdd(&st->amax_acc, 0u);
  const unsigned long long cl = atomicAdd(&st->clip_acc, 0ull);
  const unsigned long long nf = atomicAdd(&st->nonfinite_acc, 0ull);
  const unsigned long long uf = atomicAdd(&st->underflow_acc, 0ull);
  publish_and_advance(st, h, t, e, a, cl, nf, uf);
}

}  // namespace fp8q

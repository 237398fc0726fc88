// Device helpers of the scaled FP8 cast: conversion, abs-max, exponent rule
// of the per-tensor scale.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8q_internal.cuh"

namespace fp8q {

// fp32 bit patterns of the formats' largest finite values (1.75 * 2^emax).
__host__ __device__ constexpr uint32_t fmax_bits(int fmt) {
  return fmt == FP8Q_E4M3 ? 0x43E00000u /* 448 */ : 0x47600000u /* 57344 */;
}
__host__ __device__ constexpr int emax_elem(int fmt) { return fmt == FP8Q_E4M3 ? 8 : 15; }

// Two fp32 -> two FP8 bytes, round to nearest even, saturating to +-max
// (`lo` lands in the low byte).  Blackwell converts a pair per instruction.
template <int FMT>
__device__ __forceinline__ uint32_t cvt_pair(float lo, float hi) {
  unsigned short r;
  if (FMT == FP8Q_E4M3)
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t vmax_u16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Rounded-past-max test on the scaled value: E4M3's tie at 464 goes to the
// even 448, E5M2's tie at 61440 goes to the even 65536 (beyond the max).
template <int FMT>
__device__ __forceinline__ bool clips(float v) {
  return FMT == FP8Q_E4M3 ? (fabsf(v) > 464.0f) : (fabsf(v) >= 61440.0f);
}

__device__ __forceinline__ float pow2f(int e) {   // e in [-126, 127]
  return __uint_as_float((uint32_t)(127 + e) << 23);
}

// abs-bits of element j of a 16-byte load, widened to fp32 bits.
template <int DT>
__device__ __forceinline__ uint32_t elem_bits(const uint4& v, int j) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  if (DT == FP8Q_BF16) return (j & 1) ? (w[j >> 1] & 0xFFFF0000u) : (w[j >> 1] << 16);
  return w[j];
}

// Max of |x| bits over one 16-byte load.  For bf16 the result is packed
// (two u16 lanes); unpack_max turns it into fp32 bits.
template <int DT>
__device__ __forceinline__ uint32_t absmax_load(const uint4& v) {
  if (DT == FP8Q_BF16) {
    const uint32_t m = 0x7FFF7FFFu;
    return vmax_u16x2(vmax_u16x2(v.x & m, v.y & m), vmax_u16x2(v.z & m, v.w & m));
  }
  const uint32_t m = 0x7FFFFFFFu;
  return max(max(v.x & m, v.y & m), max(v.z & m, v.w & m));
}
template <int DT>
__device__ __forceinline__ uint32_t absmax_merge(uint32_t a, uint32_t b) {
  return DT == FP8Q_BF16 ? vmax_u16x2(a, b) : max(a, b);
}
template <int DT>
__device__ __forceinline__ uint32_t unpack_max(uint32_t a) {
  return DT == FP8Q_BF16 ? (max(a >> 16, a & 0xFFFFu) << 16) : a;
}

// Cast the elements of one 16-byte load scaled by s.  bf16: 8 elements -> 8
// bytes (o.x, o.y); fp32: 4 elements -> 4 bytes (o.x).
template <int DT, int FMT>
__device__ __forceinline__ uint2 cast_load(const uint4& v, float s) {
  uint2 o;
  if (DT == FP8Q_BF16) {
    const float f0 = __uint_as_float(v.x << 16) * s, f1 = __uint_as_float(v.x & 0xFFFF0000u) * s;
    const float f2 = __uint_as_float(v.y << 16) * s, f3 = __uint_as_float(v.y & 0xFFFF0000u) * s;
    const float f4 = __uint_as_float(v.z << 16) * s, f5 = __uint_as_float(v.z & 0xFFFF0000u) * s;
    const float f6 = __uint_as_float(v.w << 16) * s, f7 = __uint_as_float(v.w & 0xFFFF0000u) * s;
    o.x = cvt_pair<FMT>(f0, f1) | (cvt_pair<FMT>(f2, f3) << 16);
    o.y = cvt_pair<FMT>(f4, f5) | (cvt_pair<FMT>(f6, f7) << 16);
  } else {
    const float f0 = __uint_as_float(v.x) * s, f1 = __uint_as_float(v.y) * s;
    const float f2 = __uint_as_float(v.z) * s, f3 = __uint_as_float(v.w) * s;
    o.x = cvt_pair<FMT>(f0, f1) | (cvt_pair<FMT>(f2, f3) << 16);
    o.y = 0;
  }
  return o;
}

// Exact per-element pass over one load, taken only when some |x| of the
// chunk exceeds fmax * 2^-e or is not finite: counts the clipped elements
// and writes NaN inputs as sign|0x7F.
template <int DT, int FMT>
__device__ __forceinline__ void fix_load(const uint4& v, float s, uint2& o, uint32_t& clip,
                                         uint32_t* s_nonfinite) {
  constexpr int EPL = DT == FP8Q_BF16 ? 8 : 4;
  uint32_t nonfinite = 0;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const uint32_t b = elem_bits<DT>(v, j);
    const float f = __uint_as_float(b) * s;
    clip += clips<FMT>(f) ? 1u : 0u;
    nonfinite += (b & 0x7FFFFFFFu) >= 0x7F800000u ? 1u : 0u;
    if ((b & 0x7FFFFFFFu) > 0x7F800000u) {
      const uint32_t byte = ((b >> 31) << 7) | 0x7Fu;
      const int sh = (j & 3) * 8;
      if (j < 4) o.x = (o.x & ~(0xFFu << sh)) | (byte << sh);
      else o.y = (o.y & ~(0xFFu << sh)) | (byte << sh);
    }
  }
  // rare path: a shared-memory counter keeps the common path's registers free
  if (nonfinite) atomicAdd(s_nonfinite, nonfinite);
}

// fp32 bits of the largest |x| whose scaled value x * 2^e rounds to zero:
// half the smallest subnormal (2^-10 for E4M3, 2^-17 for E5M2; the tie goes
// to the even zero) times 2^-e; 0 when that is below the smallest fp32.
__device__ __forceinline__ uint32_t underflow_bound(int fmt, int e) {
  const int k = (fmt == FP8Q_E4M3 ? -10 : -17) - e;
  if (k >= -126) return (uint32_t)(k + 127) << 23;
  if (k >= -149) return 1u << (k + 149);
  return 0u;
}

// Inputs of one 16-byte load that underflow (0 < |x| <= bound).  bf16: two
// per word, compared in place: (B|0x8000) - a keeps bit 15 iff a <= B, and
// a + 0x7FFF sets bit 15 iff a >= 1 (no carry crosses the half-words).
template <int DT>
__device__ __forceinline__ uint32_t underflow_load(const uint4& v, uint32_t bound) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t n = 0;
  if (DT == FP8Q_BF16) {
    const uint32_t b16 = bound >> 16;
    const uint32_t bb = (b16 | (b16 << 16)) | 0x80008000u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t a = w[i] & 0x7FFF7FFFu;
      n += __popc((bb - a) & (a + 0x7FFF7FFFu) & 0x80008000u);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) n += ((w[i] & 0x7FFFFFFFu) - 1u < bound) ? 1u : 0u;
  }
  return n;
}

// Scale exponent from an amax (fp32 bits): the largest e with
// 2^e * A <= fmax * 2^-margin.  With A = mu * 2^k, mu in [1, 2) and
// fmax = 1.75 * 2^emax this is e = emax - margin - k - [mu > 1.75];
// clamped to [-126, 126].  *ok = false for a zero or non-finite A.
__device__ __forceinline__ int exp_from_amax(uint32_t a, int fmt, int margin, bool* ok) {
  a &= 0x7FFFFFFFu;
  if (a == 0u || a >= 0x7F800000u) { *ok = false; return 0; }
  *ok = true;
  const uint32_t ef = a >> 23, mf = a & 0x7FFFFFu;
  int k;
  bool gt;
  if (ef != 0u) {
    k = (int)ef - 127;
    gt = mf > 0x600000u;                       // mu > 1.75
  } else {                                     // subnormal amax
    const int lb = 31 - __clz((int)mf);
    k = lb - 149;
    gt = (mf << 2) > (7u << lb);
  }
  int e = emax_elem(fmt) - margin - k - (gt ? 1 : 0);
  return min(126, max(-126, e));
}

// Exponent for this cast from the window maximum, the previous exponent
// and the hysteresis rule (only an upward move of 1..hyst binades is held).
__device__ __forceinline__ int pick_exp(uint32_t a_w, int fmt, int margin, int hyst,
                                        int prev_e, bool has_prev) {
  bool ok;
  const int e = exp_from_amax(a_w, fmt, margin, &ok);
  if (!ok) return has_prev ? prev_e : 0;
  if (has_prev && e > prev_e && e - prev_e <= hyst) return prev_e;
  return e;
}

// fp32 bits of fmax * 2^-e (largest |x| that cannot clip), or the largest
// finite fp32 when that overflows (then only Inf / NaN exceed it).
__device__ __forceinline__ uint32_t no_clip_bound(int fmt, int e) {
  const int be = (int)(fmax_bits(fmt) >> 23) - e;
  return be >= 255 ? 0x7F7FFFFFu : fmax_bits(fmt) - ((uint32_t)e << 23);
}

}  // namespace fp8q

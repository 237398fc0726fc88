// MX (microscaling) shared-exponent rules: one power of two per 32-element
// block, stored as an E8M0 byte E + 127 ("what actually breaks low precision
// training": the OCP formula, the round-up variant, and headroom).
#pragma once

#include <stdint.h>

#include "fp8q_device.cuh"

namespace fp8q {

// Larger magnitude in one instruction: max(|a|, |b|) per bf16 lane of a
// packed pair (or of two fp32 values), the exact larger magnitude with its
// sign bit set to the XOR of the input signs, and the canonical NaN when
// either input is NaN.  The caller masks the sign bits once at the end, which
// leaves the same bits as an integer max of the masked abs bits (NaN above
// Inf above every finite value).
template <int DT>
__device__ __forceinline__ uint32_t mag_max(uint32_t a, uint32_t b) {
  uint32_t r;
  if (DT == FP8Q_BF16) {
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  } else {
    float f;
    asm("max.NaN.xorsign.abs.f32 %0, %1, %2;" : "=f"(f) : "f"(__uint_as_float(a)), "f"(__uint_as_float(b)));
    r = __float_as_uint(f);
  }
  return r;
}
// Over one 16-byte load (packed pairs for bf16; signs not yet masked).
template <int DT>
__device__ __forceinline__ uint32_t mag_load(const uint4& v) {
  return mag_max<DT>(mag_max<DT>(v.x, v.y), mag_max<DT>(v.z, v.w));
}
// Masked magnitude as fp32 bits (for bf16: the larger of the two lanes).
template <int DT>
__device__ __forceinline__ uint32_t mag_bits(uint32_t m) {
  return unpack_max<DT>(m & (DT == FP8Q_BF16 ? 0x7FFF7FFFu : 0x7FFFFFFFu));
}

// Shared exponent of a block from its amax bits m (finite), per rule:
//   floor (OCP): E = floor(log2 A) - emax_elem
//   ceil:        smallest E with A * 2^-E <= fmax; with A = mu * 2^k this is
//                k - emax_elem + [mu > 1.75]   (fmax = 1.75 * 2^emax_elem)
//   nearest:     E nearest to log2(A / fmax):   k - emax_elem - [mu < 1.75/sqrt 2],
//                tested exactly as M^2 < 49 * 2^41 on the 24-bit significand M,
//                i.e. M <= isqrt(49 * 2^41 - 1) = 10380372 (0x9E6454)
// then + headroom, clamped to [-127, 127]; a zero block gets -127.
template <int FMT>
__device__ __forceinline__ int block_exp(uint32_t m, int rule, int headroom) {
  if (m == 0u) return -127;
  int k;
  uint32_t M;
  if (m >> 23) {
    k = (int)(m >> 23) - 127;
    M = 0x800000u | (m & 0x7FFFFFu);
  } else {
    const int lb = 31 - __clz((int)m);
    k = lb - 149;
    M = m << (23 - lb);
  }
  int E = k - emax_elem(FMT);
  if (rule == FP8Q_MX_CEIL) E += (M > 0xE00000u) ? 1 : 0;
  else if (rule == FP8Q_MX_NEAREST) E -= (M <= 0x9E6454u) ? 1 : 0;
  return min(127, max(-127, E + headroom));
}

// Finite bf16 / fp32 block maxima have k <= 127, so E <= 127 - emax_elem +
// 1 (ceil) + headroom.  The casts scale by 2^-E as the normal fp32 number
// with exponent field 127 - E, which needs E <= 126: headroom is therefore
// capped (the C ABI rejects more than kMaxHeadroom).
constexpr int kMaxHeadroom = 4;
static_assert(127 - 8 + 1 + kMaxHeadroom <= 126, "2^-E must stay a normal fp32 number");

// Can a finite block with max |x| bits m and shared exponent E hold a clipped
// element?  Only if its scaled maximum m * 2^-E passes fmax, i.e. m exceeds
// fmax * 2^E (never when that is beyond the fp32 range).
template <int FMT>
__device__ __forceinline__ bool mx_block_may_clip(uint32_t m, int E) {
  const int be = (int)(fmax_bits(FMT) >> 23) + E;
  return be < 255 && m > fmax_bits(FMT) + ((uint32_t)E << 23);
}

}  // namespace fp8q

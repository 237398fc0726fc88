// MX (microscaling) shared-exponent rules: one power of two per 32-element
// block, stored as an E8M0 byte E + 127 ("what actually breaks low precision
// training": the OCP formula, the round-up variant, and headroom).
#pragma once

#include <stdint.h>

#include "fp8q_device.cuh"

namespace fp8q {

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

}  // namespace fp8q

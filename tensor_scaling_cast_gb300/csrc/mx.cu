// MX block-scaled cast: 32 consecutive elements of a row share one power of
// two, E = floor(log2(block amax)) - emax_elem (+ headroom), stored as an
// E8M0 byte E + 127 ("what actually breaks low precision training", "What
// the measurements said": the OCP formula, and one extra bit of headroom).
//
// Thread mapping: each lane owns one 16-byte load (8 bf16 or 4 fp32), so a
// warp-wide load is 512 contiguous bytes and a 32-element block spans 4
// (bf16) or 8 (fp32) consecutive lanes.  The block amax is an integer max of
// abs bits finished with 2-3 xor-shuffles; E comes from the exponent field
// (leading-bit position for subnormals).  Blocks are independent, so there
// is no cross-CTA step besides one atomic add of the clipped count.
#include <cuda_runtime.h>

#include "fp8q_device.cuh"
#include "fp8q_internal.cuh"

namespace fp8q {

template <int DT, int FMT>
__global__ void __launch_bounds__(kThreads, 4) mx_kernel(const char* __restrict__ x, int64_t nelem,
                                                      uint8_t* __restrict__ q,
                                                      uint8_t* __restrict__ e8m0,
                                                      unsigned long long* clipped, int headroom) {
  constexpr int EPL = DT == FP8Q_BF16 ? 8 : 4;    // elements per lane-load
  constexpr int ESZ = DT == FP8Q_BF16 ? 2 : 4;
  constexpr int LPB = 32 / EPL;                   // lanes per 32-element block
  constexpr int64_t TILE = (int64_t)kThreads * kUnroll * EPL;
  __shared__ uint32_t red_c[kThreads / 32];
  const int lane = threadIdx.x & 31;
  uint32_t lclip = 0;
  const int64_t ntiles = (nelem + TILE - 1) / TILE;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t base = tile * TILE;
    uint4 r[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t e0 = base + (int64_t)(u * kThreads + threadIdx.x) * EPL;
      // nelem is a multiple of 32, so a lane-load is entirely in or out
      r[u] = e0 < nelem ? __ldcs(reinterpret_cast<const uint4*>(x + e0 * ESZ)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t e0 = base + (int64_t)(u * kThreads + threadIdx.x) * EPL;
      uint32_t m = unpack_max<DT>(absmax_load<DT>(r[u]));
#pragma unroll
      for (int o = 1; o < LPB; o <<= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      uint2 out;
      uint32_t ebyte;
      if (m >= 0x7F800000u) {                      // NaN or Inf in the block
        ebyte = 0xFFu;
        uint32_t w[2] = {0u, 0u};
#pragma unroll
        for (int j = 0; j < EPL; ++j)
          w[j >> 2] |= ((((elem_bits<DT>(r[u], j) >> 31) << 7) | 0x7Fu) << ((j & 3) * 8));
        out = make_uint2(w[0], w[1]);
      } else {
        int E;
        if (m == 0u) {
          E = -127;
        } else {
          const int fl = (m >> 23) ? (int)(m >> 23) - 127 : (31 - __clz((int)m)) - 149;
          E = min(127, max(-127, fl - emax_elem(FMT) + headroom));
        }
        ebyte = (uint32_t)(E + 127);
        const float s = __uint_as_float((uint32_t)(127 - E) << 23);   // 2^-E
        out = cast_load<DT, FMT>(r[u], s);
        // per-element count only for blocks whose scaled max passes fmax
        const int be = (int)(fmax_bits(FMT) >> 23) + E;
        const uint32_t bound = be >= 255 ? 0x7F7FFFFFu : fmax_bits(FMT) + ((uint32_t)E << 23);
        if (m > bound) {
#pragma unroll
          for (int j = 0; j < EPL; ++j)
            lclip += clips<FMT>(__uint_as_float(elem_bits<DT>(r[u], j)) * s) ? 1u : 0u;
        }
      }
      if (e0 < nelem) {
        if (DT == FP8Q_BF16) __stcs(reinterpret_cast<uint2*>(q + e0), out);
        else __stcs(reinterpret_cast<unsigned int*>(q + e0), out.x);
        if ((lane & (LPB - 1)) == 0) e8m0[e0 >> 5] = (uint8_t)ebyte;
      }
    }
  }
  if (clipped) {
    lclip = __reduce_add_sync(0xFFFFFFFFu, lclip);
    if (lane == 0) red_c[threadIdx.x >> 5] = lclip;
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned long long tot = 0;
      for (int i = 0; i < kThreads / 32; ++i) tot += red_c[i];
      if (tot) atomicAdd(clipped, tot);
    }
  }
}

template <int DT, int FMT>
static cudaError_t launch_mx_t(const void* x, int64_t nelem, int headroom, uint8_t* q, uint8_t* e8m0,
                               unsigned long long* clipped, cudaStream_t s, int* launches) {
  constexpr int EPL = DT == FP8Q_BF16 ? 8 : 4;
  constexpr int64_t TILE = (int64_t)kThreads * kUnroll * EPL;
  static int occ = 0;
  if (occ == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, mx_kernel<DT, FMT>, kThreads, 0) != cudaSuccess || occ < 1)
      occ = 1;
  }
  const int64_t ntiles = (nelem + TILE - 1) / TILE;
  long long grid = (long long)sm_count(device_of_current()) * occ;
  if (grid > ntiles) grid = ntiles;
  if (grid < 1) grid = 1;
  mx_kernel<DT, FMT><<<(unsigned)grid, kThreads, 0, s>>>(reinterpret_cast<const char*>(x), nelem, q, e8m0,
                                                        clipped, headroom);
  ++*launches;
  return cudaGetLastError();
}

cudaError_t launch_mx(const void* x, int dtype, int64_t nelem, int format, int headroom, uint8_t* q,
                      uint8_t* e8m0, unsigned long long* clipped, cudaStream_t s, int* launches) {
  if (dtype == FP8Q_BF16)
    return format == FP8Q_E4M3 ? launch_mx_t<FP8Q_BF16, FP8Q_E4M3>(x, nelem, headroom, q, e8m0, clipped, s, launches)
                               : launch_mx_t<FP8Q_BF16, FP8Q_E5M2>(x, nelem, headroom, q, e8m0, clipped, s, launches);
  return format == FP8Q_E4M3 ? launch_mx_t<FP8Q_F32, FP8Q_E4M3>(x, nelem, headroom, q, e8m0, clipped, s, launches)
                             : launch_mx_t<FP8Q_F32, FP8Q_E5M2>(x, nelem, headroom, q, e8m0, clipped, s, launches);
}

}  // namespace fp8q

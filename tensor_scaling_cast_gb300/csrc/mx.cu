// MX block-scaled cast: 32 consecutive elements of a row share one power of
// two, E = floor(log2(block amax)) - emax_elem (+ headroom), stored as an
// E8M0 byte E + 127 ("what actually breaks low precision training", "What
// the measurements said": the OCP formula, and one extra bit of headroom).
//
// Thread mapping: each lane owns one 16-byte load (8 bf16 or 4 fp32), so a
// warp-wide load is 512 contiguous bytes and a 32-element block spans 4
// (bf16) or 8 (fp32) consecutive lanes.  The block amax is a magnitude max
// over the lane's load (one max.NaN.xorsign.abs per pair of words, the
// signs masked at the end) finished with 2-3 xor-shuffles; E comes from the
// exponent field (leading-bit position for subnormals).  Blocks are
// independent, so there is no cross-CTA step besides one atomic add of the
// clipped count.
#include <cuda.h>
#include <cuda_runtime.h>

#include "fp8q_device.cuh"
#include "fp8q_internal.cuh"
#include "mx_device.cuh"
#include "tma.cuh"
#include "warp_tiles.cuh"

namespace fp8q {

// Lane-loads per thread per tile of the row-wise kernel: 4 (16 KiB tiles)
// measured 2-3% faster than the grouped cast's 8 on bf16 [16384, 8192].
constexpr int kMxUnroll = 4;

template <int DT, int FMT>
__global__ void __launch_bounds__(kThreads, 4) mx_kernel(const char* __restrict__ x, int64_t nelem,
                                                      uint8_t* __restrict__ q,
                                                      uint8_t* __restrict__ e8m0,
                                                      unsigned long long* clipped, int headroom,
                                                      int rule) {
  constexpr int EPL = DT == FP8Q_BF16 ? 8 : 4;    // elements per lane-load
  constexpr int ESZ = DT == FP8Q_BF16 ? 2 : 4;
  constexpr int LPB = 32 / EPL;                   // lanes per 32-element block
  constexpr int64_t TILE = (int64_t)kThreads * kMxUnroll * EPL;
  __shared__ uint32_t red_c[kThreads / 32];
  const int lane = threadIdx.x & 31;
  uint32_t lclip = 0;
  const int64_t ntiles = (nelem + TILE - 1) / TILE;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t base = tile * TILE;
    uint4 r[kMxUnroll];
#pragma unroll
    for (int u = 0; u < kMxUnroll; ++u) {
      const int64_t e0 = base + (int64_t)(u * kThreads + threadIdx.x) * EPL;
      // nelem is a multiple of 32, so a lane-load is entirely in or out
      r[u] = e0 < nelem ? __ldcs(reinterpret_cast<const uint4*>(x + e0 * ESZ)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kMxUnroll; ++u) {
      const int64_t e0 = base + (int64_t)(u * kThreads + threadIdx.x) * EPL;
      uint32_t m = mag_bits<DT>(mag_load<DT>(r[u]));
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
        const int E = block_exp<FMT>(m, rule, headroom);
        ebyte = (uint32_t)(E + 127);
        const float s = __uint_as_float((uint32_t)(127 - E) << 23);   // 2^-E
        out = cast_load<DT, FMT>(r[u], s);
        // per-element count only for blocks whose scaled max passes fmax
        if (mx_block_may_clip<FMT>(m, E)) {
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
static cudaError_t launch_mx_t(const void* x, int64_t nelem, int headroom, int rule, uint8_t* q,
                               uint8_t* e8m0, unsigned long long* clipped, cudaStream_t s,
                               int* launches) {
  constexpr int EPL = DT == FP8Q_BF16 ? 8 : 4;
  constexpr int64_t TILE = (int64_t)kThreads * kMxUnroll * EPL;
  int occ = 1;
  cudaError_t oe = kernel_occupancy(reinterpret_cast<const void*>(mx_kernel<DT, FMT>), kThreads, 0, &occ);
  if (oe != cudaSuccess) return oe;
  const int64_t ntiles = (nelem + TILE - 1) / TILE;
  long long grid = (long long)sm_count(device_of_current()) * occ;
  if (grid > ntiles) grid = ntiles;
  if (grid < 1) grid = 1;
  mx_kernel<DT, FMT><<<(unsigned)grid, kThreads, 0, s>>>(reinterpret_cast<const char*>(x), nelem, q, e8m0,
                                                        clipped, headroom, rule);
  ++*launches;
  return cudaGetLastError();
}

cudaError_t launch_mx(const void* x, int dtype, int64_t nelem, int format, int headroom, int rule,
                      uint8_t* q, uint8_t* e8m0, unsigned long long* clipped, cudaStream_t s,
                      int* launches) {
  if (dtype == FP8Q_BF16)
    return format == FP8Q_E4M3
               ? launch_mx_t<FP8Q_BF16, FP8Q_E4M3>(x, nelem, headroom, rule, q, e8m0, clipped, s, launches)
               : launch_mx_t<FP8Q_BF16, FP8Q_E5M2>(x, nelem, headroom, rule, q, e8m0, clipped, s, launches);
  return format == FP8Q_E4M3
             ? launch_mx_t<FP8Q_F32, FP8Q_E4M3>(x, nelem, headroom, rule, q, e8m0, clipped, s, launches)
             : launch_mx_t<FP8Q_F32, FP8Q_E5M2>(x, nelem, headroom, rule, q, e8m0, clipped, s, launches);
}

// ---- column-wise blocks ------------------------------------------------------
//
// Blocks of 32 consecutive rows of one column (the operand layout a backward
// matmul reads along its first dimension), q and e8m0 row-major like x.
// Each warp runs the per-warp TMA pipeline of warp_tiles.cuh over 32-row x
// 128-byte sub-tiles.  Lane l takes bf16 columns 2l, 2l + 1 (one 32-bit
// shared word per row) or fp32 column l: the block max, E and the cast of
// its 32 values all stay in the lane.  The lane's bytes go row by row into a
// swizzled staging tile (a bf16 lane writes one 16-bit pair per row, built
// with byte permutes) that a TMA tiled store copies to q; the E8M0 bytes of a
// sub-tile are one coalesced row segment.

// Sixteen two-stage warps per SM, in one CTA (adjacent column tiles), when
// blocks may clip (the exact per-element count needs the warps); two CTAs
// of four three-stage warps per SM for a clip-free cast (mx_clip_free),
// which is memory-bound.  Column strips first; the L2 fetches 128 bytes per
// input request.
using ColCfg = TpCfg<2, 2, 1, true, 2048, 1, true, 16>;
using ColClipFreeCfg = TpCfg<3, 2, 1, true, 2048, 2, false>;
constexpr int kColL2Promotion = 128;

static __device__ unsigned int g_wait_timeouts;

template <int DT, int FMT, class C>
__global__ void __launch_bounds__(C::kThreads, C::kMinBlocks) mx_colwise_kernel(
    const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap qmap, int64_t rows,
    int64_t cols, uint8_t* __restrict__ e8m0, unsigned long long* clipped, int headroom, int rule) {
  constexpr int TILE_C = TileGeom<DT>::TILE_C;
  extern __shared__ __align__(1024) uint4 dyn_smem[];
  __shared__ __align__(8) uint64_t full[C::kWarps][C::kStages];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t ctiles = (uint32_t)((cols + TILE_C - 1) / TILE_C);
  uint8_t* region = warp_region<C>(dyn_smem, warp);
  WarpPipe<C> pipe;
  pipe.setup(&tmap, reinterpret_cast<uint4*>(region), full[warp], (uint32_t)(rows / 32), ctiles, TILE_C,
             &g_wait_timeouts);
  const OutStage<C> out{region + C::kStages * kWTileBytes};
  pipe.start();
  uint32_t clip = 0;
  for (uint32_t j = 0; pipe.valid(pipe.cur); ++j) {
    if (!pipe.wait(j)) {
      out.drain();
      return;
    }
    const uint4* tile = pipe.tile(j);
    const int64_t r0 = pipe.r0(), c0 = pipe.c0();
    out.acquire();
    uint8_t* ob = out.buf(j);
    uint8_t* e8 = e8m0 + (r0 >> 5) * cols;
    uint32_t w[32];
    if (DT == FP8Q_BF16) {
      const int64_t c = c0 + 2 * lane;
      if (c < cols) {
        load_column_words(tile, lane, w);
        const uint32_t pm = tree_absmax32<true>(w);
        uint32_t o0[8], o1[8];
        const uint32_t e0 = mx_column<FMT, 0, C::kClipCount>(w, pm << 16, rule, headroom, clip, o0);
        const uint32_t e1 = mx_column<FMT, 1, C::kClipCount>(w, pm & 0xFFFF0000u, rule, headroom, clip, o1);
#pragma unroll
        for (int m = 0; m < 8; ++m) {               // rows 4m .. 4m + 3: (column 2l, column 2l + 1) pairs
          const uint32_t lo = __byte_perm(o0[m], o1[m], 0x5140);
          const uint32_t hi = __byte_perm(o0[m], o1[m], 0x7362);
          *reinterpret_cast<uint16_t*>(ob + staged_byte<64>(4 * m, 2 * lane)) = (uint16_t)lo;
          *reinterpret_cast<uint16_t*>(ob + staged_byte<64>(4 * m + 1, 2 * lane)) = (uint16_t)(lo >> 16);
          *reinterpret_cast<uint16_t*>(ob + staged_byte<64>(4 * m + 2, 2 * lane)) = (uint16_t)hi;
          *reinterpret_cast<uint16_t*>(ob + staged_byte<64>(4 * m + 3, 2 * lane)) = (uint16_t)(hi >> 16);
        }
        uint8_t* e = e8 + c;
        if ((reinterpret_cast<uintptr_t>(e) & 1u) == 0) {
          *reinterpret_cast<uint16_t*>(e) = (uint16_t)(e0 | (e1 << 8));
        } else {
          e[0] = (uint8_t)e0;
          e[1] = (uint8_t)e1;
        }
      }
    } else {
      const int64_t c = c0 + lane;
      if (c < cols) {
        load_column_words(tile, lane, w);
        uint32_t o[8];
        e8[c] = (uint8_t)mx_column<FMT, 2, C::kClipCount>(w, tree_absmax32<false>(w), rule, headroom, clip, o);
#pragma unroll
        for (int k = 0; k < 32; ++k) ob[staged_byte<32>(k, lane)] = (uint8_t)(o[k >> 2] >> (8 * (k & 3)));
      }
    }
    out.publish(j, &qmap, nullptr, r0, c0);
    pipe.release();
  }
  out.drain();
  clip = __reduce_add_sync(0xFFFFFFFFu, clip);
  if (clipped && lane == 0 && clip) atomicAdd(clipped, (unsigned long long)clip);
}

template <int DT, int FMT, class C>
static cudaError_t launch_mx_col_c(const void* x, int64_t rows, int64_t cols, int headroom, int rule,
                                   uint8_t* q, uint8_t* e8m0, unsigned long long* clipped,
                                   cudaStream_t s, int* launches) {
  constexpr int TILE_C = TileGeom<DT>::TILE_C;
  auto kern = mx_colwise_kernel<DT, FMT, C>;
  const int64_t ctiles = (cols + TILE_C - 1) / TILE_C;
  if ((rows / 32) * ctiles >= (int64_t(1) << 31)) return cudaErrorInvalidValue;   // 32-bit tile counts
  int occ = 1;
  cudaError_t e = kernel_occupancy(reinterpret_cast<const void*>(kern), C::kThreads, C::kSmemBytes, &occ);
  if (e != cudaSuccess) return e;
  if (C::kMaxCtasPerSm > 0 && occ > C::kMaxCtasPerSm) occ = C::kMaxCtasPerSm;
  CUtensorMap in, qm;
  e = encode_tile_map(&in, x, DT == FP8Q_BF16, rows, cols, TILE_C, true, kColL2Promotion);
  if (e == cudaSuccess) e = encode_byte_map(&qm, q, rows, cols, TILE_C, 32, TILE_C);
  if (e != cudaSuccess) return e;
  const long long need = ((rows / 32) * ctiles + C::kWarps - 1) / C::kWarps;
  long long grid = (long long)sm_count(device_of_current()) * occ;
  if (grid > need) grid = need;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, C::kThreads, C::kSmemBytes, s>>>(in, qm, rows, cols, e8m0, clipped, headroom, rule);
  ++*launches;
  return cudaGetLastError();
}

template <int DT, int FMT>
static cudaError_t launch_mx_col_t(const void* x, int64_t rows, int64_t cols, int headroom, int rule,
                                   uint8_t* q, uint8_t* e8m0, unsigned long long* clipped, cudaStream_t s,
                                   int* launches) {
  return mx_clip_free(rule, headroom)
             ? launch_mx_col_c<DT, FMT, ColClipFreeCfg>(x, rows, cols, headroom, rule, q, e8m0, clipped, s, launches)
             : launch_mx_col_c<DT, FMT, ColCfg>(x, rows, cols, headroom, rule, q, e8m0, clipped, s, launches);
}

cudaError_t launch_mx_colwise(const void* x, int dtype, int64_t rows, int64_t cols, int format,
                              int headroom, int rule, uint8_t* q, uint8_t* e8m0,
                              unsigned long long* clipped, cudaStream_t s, int* launches) {
  if (dtype == FP8Q_BF16)
    return format == FP8Q_E4M3
               ? launch_mx_col_t<FP8Q_BF16, FP8Q_E4M3>(x, rows, cols, headroom, rule, q, e8m0, clipped, s, launches)
               : launch_mx_col_t<FP8Q_BF16, FP8Q_E5M2>(x, rows, cols, headroom, rule, q, e8m0, clipped, s, launches);
  return format == FP8Q_E4M3
             ? launch_mx_col_t<FP8Q_F32, FP8Q_E4M3>(x, rows, cols, headroom, rule, q, e8m0, clipped, s, launches)
             : launch_mx_col_t<FP8Q_F32, FP8Q_E5M2>(x, rows, cols, headroom, rule, q, e8m0, clipped, s, launches);
}

// Diagnostic: one warp waits on a barrier that nothing arms or completes.
// The bounded wait gives up at its deadline and the timeout is counted, as
// a stalled tile would be; nothing faults and nothing spins without end.
__global__ void pipeline_selftest_kernel() {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  const bool ok = mbar_wait(&bar, 0u);
  if (__syncthreads_or(!ok) && threadIdx.x == 0) atomicAdd(&g_wait_timeouts, 1u);
}

cudaError_t launch_pipeline_selftest(cudaStream_t s, int* launches) {
  pipeline_selftest_kernel<<<1, 32, 0, s>>>();
  ++*launches;
  return cudaGetLastError();
}

cudaError_t read_wait_timeouts(unsigned int* count) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(count, g_wait_timeouts, sizeof(unsigned int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof(unsigned int));
  return e;
}

}  // namespace fp8q

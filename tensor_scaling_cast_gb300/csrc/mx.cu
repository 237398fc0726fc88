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
#include <cuda.h>
#include <cuda_runtime.h>

#include "fp8q_device.cuh"
#include "tma.cuh"
#include "fp8q_internal.cuh"

namespace fp8q {

template <int DT, int FMT>
__global__ void __launch_bounds__(kThreads, 4) mx_kernel(const char* __restrict__ x, int64_t nelem,
                                                      uint8_t* __restrict__ q,
                                                      uint8_t* __restrict__ e8m0,
                                                      unsigned long long* clipped, int headroom,
                                                      int rule) {
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
        const int E = block_exp<FMT>(m, rule, headroom);
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
static cudaError_t launch_mx_t(const void* x, int64_t nelem, int headroom, int rule, uint8_t* q,
                               uint8_t* e8m0, unsigned long long* clipped, cudaStream_t s,
                               int* launches) {
  constexpr int EPL = DT == FP8Q_BF16 ? 8 : 4;
  constexpr int64_t TILE = (int64_t)kThreads * kUnroll * EPL;
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
// matmul reads along its first dimension).  Tiles of 32 rows x TILE_C columns
// (16 KiB: 256 bf16 or 128 fp32 columns) stream into shared memory through a
// 4-stage TMA pipeline (cp.async.bulk.tensor.2d, one mbarrier per stage,
// thread 0 issuing three tiles ahead), so loads stay in flight while the CTA
// works on the current tile:
//   1. each thread takes the max over 4 rows of its 16-byte column group;
//   2. one thread per column combines the 8 partial maxima, computes E,
//      writes the E8M0 byte (a warp writes 32 consecutive bytes) and
//      publishes E in shared memory;
//   3. each thread casts its 4 rows x EPL columns and stores them row-major
//      (a warp covers one 256-byte (bf16) row segment per store).
// Every barrier wait is bounded; a tile that does not arrive in time is
// counted in g_wait_timeouts (fp8q_pipeline_status) and the CTA stops.

constexpr int kColStages = 4;
constexpr int kColTileBytes = 32 * 32 * 16;            // 32 rows x 32 16-byte groups

static __device__ unsigned int g_wait_timeouts;

template <int DT, int FMT>
__global__ void __launch_bounds__(kThreads, 2) mx_colwise_kernel(
    const __grid_constant__ CUtensorMap tmap, int64_t rows, int64_t cols, uint8_t* __restrict__ q,
    uint8_t* __restrict__ e8m0, unsigned long long* clipped, int headroom, int rule) {
  constexpr int EPL = DT == FP8Q_BF16 ? 8 : 4;      // columns per 16-byte group
  constexpr int GROUPS = 32;                         // 16-byte groups per tile row
  constexpr int TILE_C = GROUPS * EPL;               // 256 (bf16) / 128 (fp32) columns
  extern __shared__ __align__(1024) uint4 dyn_smem[];
  // kColStages tiles [32][GROUPS], base rounded up to 1024 bytes (TMA needs
  // at least 128-byte aligned destinations; the launch adds 1 KiB of slack)
  uint4* const stage_mem = reinterpret_cast<uint4*>(
      reinterpret_cast<char*>(dyn_smem) + ((1024u - (smem_addr(dyn_smem) & 1023u)) & 1023u));
  __shared__ __align__(8) uint64_t full[kColStages];
  __shared__ uint4 part[8][GROUPS];                  // per row-group packed maxima
  __shared__ __align__(8) signed char s_e[TILE_C];   // E per column, -128 = NaN/Inf block
  __shared__ __align__(8) unsigned char s_flag[TILE_C];  // 1: block max passes fmax, 2: not finite
  __shared__ uint32_t red_c[kThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t col_tiles = (cols + TILE_C - 1) / TILE_C;
  const int64_t ntiles = (rows / 32) * col_tiles;
  const int64_t mine = ntiles > (int64_t)blockIdx.x ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  auto issue = [&](int64_t j) {                      // thread 0: tile j of this CTA
    const int64_t t = blockIdx.x + j * (int64_t)gridDim.x;
    const int st = (int)(j % kColStages);
    mbar_arrive_expect_tx(&full[st], kColTileBytes);
    tma_load_2d(stage_mem + st * 32 * GROUPS, &tmap, &full[st], (int)((t % col_tiles) * TILE_C),
                (int)((t / col_tiles) * 32));
  };
  if (tid == 0) {
    for (int i = 0; i < kColStages; ++i) mbar_init(&full[i], 1);
    fence_barrier_init();
    prefetch_tensormap(&tmap);
  }
  __syncthreads();
  if (tid == 0)
    for (int64_t j = 0; j < kColStages - 1 && j < mine; ++j) issue(j);

  uint32_t lclip = 0;
  for (int64_t j = 0; j < mine; ++j) {
    // refill the stage every thread finished with in the previous iteration
    if (tid == 0 && j + kColStages - 1 < mine) {
      fence_proxy_async();
      issue(j + kColStages - 1);
    }
    const int st = (int)(j % kColStages);
    const bool ok = mbar_wait(&full[st], (uint32_t)((j / kColStages) & 1));
    const uint4(*tile)[GROUPS] = reinterpret_cast<const uint4(*)[GROUPS]>(stage_mem + st * 32 * GROUPS);
    const int64_t t = blockIdx.x + j * (int64_t)gridDim.x;
    const int64_t r0 = (t / col_tiles) * 32, c0 = (t % col_tiles) * TILE_C;

    // 1. partial maxima: thread (warp w, lane g) covers rows 4w..4w+3 of group g
    uint32_t pm[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = tile[4 * warp + i][lane];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (DT == FP8Q_BF16) pm[k] = vmax_u16x2(pm[k], w[k] & 0x7FFF7FFFu);
        else pm[k] = max(pm[k], w[k] & 0x7FFFFFFFu);
      }
    }
    part[warp][lane] = make_uint4(pm[0], pm[1], pm[2], pm[3]);
    if (__syncthreads_or(!ok)) {                     // a tile did not arrive in time
      if (tid == 0) {
        atomicAdd(&g_wait_timeouts, 1u);
        for (int64_t k = j; k < j + kColStages - 1 && k < mine; ++k)   // bounded drain
          mbar_wait(&full[k % kColStages], (uint32_t)((k / kColStages) & 1));
      }
      return;
    }
    // 2. one thread per column: final max, exponent, E8M0 byte
    if (tid < TILE_C) {
      const int g = tid / EPL, c = tid % EPL;
      const int word = DT == FP8Q_BF16 ? (c >> 1) : c;
      uint32_t m = 0;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        uint32_t v = reinterpret_cast<const uint32_t*>(&part[w][g])[word];
        if (DT == FP8Q_BF16) v = (c & 1) ? (v & 0xFFFF0000u) : (v << 16);
        m = max(m, v);
      }
      int E;
      uint32_t byte, flag;
      if (m >= 0x7F800000u) {                        // NaN / Inf block
        E = -128;
        byte = 0xFFu;
        flag = 2u;
      } else {
        E = block_exp<FMT>(m, rule, headroom);
        byte = (uint32_t)(E + 127);
        const int be = (int)(fmax_bits(FMT) >> 23) + E;
        flag = (be < 255 && m > fmax_bits(FMT) + ((uint32_t)E << 23)) ? 1u : 0u;
      }
      s_e[tid] = (signed char)E;
      s_flag[tid] = (unsigned char)flag;
      if (c0 + tid < cols) e8m0[(r0 / 32) * cols + c0 + tid] = (uint8_t)byte;
    }
    __syncthreads();
    // 3. cast 4 rows x EPL columns, row-major stores.  Columns whose block
    // max stays within fmax need no per-element check (the common case).
    const int64_t cbase = c0 + (int64_t)lane * EPL;
    if (cbase < cols) {
      signed char eb[EPL];
      uint32_t any_flag;
      if (DT == FP8Q_BF16) {
        *reinterpret_cast<uint2*>(eb) = *reinterpret_cast<const uint2*>(&s_e[lane * EPL]);
        const uint2 fw = *reinterpret_cast<const uint2*>(&s_flag[lane * EPL]);
        any_flag = fw.x | fw.y;
      } else {
        *reinterpret_cast<uint32_t*>(eb) = *reinterpret_cast<const uint32_t*>(&s_e[lane * EPL]);
        any_flag = *reinterpret_cast<const uint32_t*>(&s_flag[lane * EPL]);
      }
      // a column below its bound cannot clip, so on a flagged tile the clip
      // test can run on every element; NaN / Inf columns are rare
      const bool count_clips = (any_flag & 0x01010101u) != 0u;
      const bool nonfinite = (any_flag & 0x02020202u) != 0u;
      float sc[EPL];
#pragma unroll
      for (int k = 0; k < EPL; ++k)
        sc[k] = __uint_as_float((uint32_t)(127 - (eb[k] == -128 ? 0 : (int)eb[k])) << 23);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = 4 * warp + i;
        const uint4 v = tile[r][lane];
        float f[EPL];
#pragma unroll
        for (int k = 0; k < EPL; ++k) f[k] = __uint_as_float(elem_bits<DT>(v, k)) * sc[k];
        uint32_t ob[2] = {0u, 0u};
#pragma unroll
        for (int k = 0; k < EPL; k += 2) ob[k >> 2] |= cvt_pair<FMT>(f[k], f[k + 1]) << ((k & 3) * 8);
        if (count_clips) {
#pragma unroll
          for (int k = 0; k < EPL; ++k) lclip += (eb[k] != -128 && clips<FMT>(f[k])) ? 1u : 0u;
        }
        if (nonfinite) {
#pragma unroll
          for (int k = 0; k < EPL; ++k) {
            if (eb[k] == -128) {                     // NaN / Inf block: sign|0x7F
              const uint32_t byte = ((elem_bits<DT>(v, k) >> 31) << 7) | 0x7Fu;
              const int sh = (k & 3) * 8;
              ob[k >> 2] = (ob[k >> 2] & ~(0xFFu << sh)) | (byte << sh);
            }
          }
        }
        uint8_t* dst = q + (r0 + r) * cols + cbase;
        if (DT == FP8Q_BF16) __stcs(reinterpret_cast<uint2*>(dst), make_uint2(ob[0], ob[1]));
        else __stcs(reinterpret_cast<unsigned int*>(dst), ob[0]);
      }
    }
    __syncthreads();                                  // stage / part / s_e reuse
  }
  if (clipped) {
    lclip = __reduce_add_sync(0xFFFFFFFFu, lclip);
    if (lane == 0) red_c[warp] = lclip;
    __syncthreads();
    if (tid == 0) {
      unsigned long long tot = 0;
      for (int i = 0; i < kThreads / 32; ++i) tot += red_c[i];
      if (tot) atomicAdd(clipped, tot);
    }
  }
}

template <int DT, int FMT>
static cudaError_t launch_mx_col_t(const void* x, int64_t rows, int64_t cols, int headroom, int rule,
                                   uint8_t* q, uint8_t* e8m0, unsigned long long* clipped,
                                   cudaStream_t s, int* launches) {
  constexpr int EPL = DT == FP8Q_BF16 ? 8 : 4;
  constexpr int TILE_C = 32 * EPL;
  constexpr int SMEM = kColStages * kColTileBytes + 1024;
  auto kern = mx_colwise_kernel<DT, FMT>;
  int occ = 1;
  cudaError_t oe = kernel_occupancy(reinterpret_cast<const void*>(kern), kThreads, SMEM, &occ);
  if (oe != cudaSuccess) return oe;
  CUtensorMap map;
  cudaError_t me = encode_tile_map(&map, x, DT == FP8Q_BF16, rows, cols, TILE_C);
  if (me != cudaSuccess) return me;
  const int64_t ntiles = (rows / 32) * ((cols + TILE_C - 1) / TILE_C);
  long long grid = (long long)sm_count(device_of_current()) * occ;
  if (grid > ntiles) grid = ntiles;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, kThreads, SMEM, s>>>(map, rows, cols, q, e8m0, clipped, headroom, rule);
  ++*launches;
  return cudaGetLastError();
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

// Fused cast + transpose: the row-major 8-bit tensor and its transpose from
// one read of x, for matmuls that need both operands cast ("what actually
// breaks low precision training": real low-precision training casts both
// operands of the backward matmuls).
//
//   cast_transpose_kernel  per-tensor scale (the handle's window / smoothed /
//                          current-scaling exponent): q [rows, cols] and
//                          qt [cols, rows], one amax / clipped count, the
//                          same cross-CTA ticket finish as the grouped cast;
//   mx_dual_kernel         MX: row-wise 32-blocks -> q_row + e8m0_row
//                          [rows, cols/32]; column-wise 32-blocks written
//                          transposed -> q_colT [cols, rows] + e8m0_colT
//                          [cols, rows/32] (the row-wise MX layout of x^T).
//
// Both stream 32-row tiles (256 bf16 / 128 fp32 columns, 16 KiB) through a
// 4-stage TMA pipeline (cp.async.bulk.tensor.2d + mbarrier, bounded waits).
// Per tile:
//   A. row pass: in 4 (bf16) / 8 (fp32) rounds each lane takes one 16-byte
//      group of a tile row (a warp reads 512 contiguous bytes of shared
//      memory: no bank conflicts) and writes its 8 / 4 bytes to the
//      row-major output (a warp writes 256 / 128 contiguous bytes);
//   B. column pass: one thread per column reads its 32 values (2- or 4-byte
//      shared loads, consecutive lanes on consecutive columns) and writes 32
//      contiguous bytes of the transposed output.
#include <cuda.h>
#include <cuda_runtime.h>

#include "fp8q_device.cuh"
#include "fp8q_internal.cuh"
#include "state.cuh"
#include "tma.cuh"

namespace fp8q {

constexpr int kTpStages = 4;

static __device__ unsigned int g_tp_wait_timeouts;   // see fp8q_pipeline_status

__device__ __forceinline__ void note_wait_timeout() { atomicAdd(&g_tp_wait_timeouts, 1u); }

cudaError_t read_tp_wait_timeouts(unsigned int* count) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(count, g_tp_wait_timeouts, sizeof(unsigned int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_tp_wait_timeouts, &zero, sizeof(unsigned int));
  return e;
}
constexpr int kTpTileBytes = 32 * 512;                 // 32 rows x 512 bytes
constexpr int kTpThreads = 256;

template <int DT>
struct TileGeom {
  static constexpr int EPL = DT == FP8Q_BF16 ? 8 : 4;   // elements per 16-byte group
  static constexpr int TILE_C = 32 * EPL;               // 256 / 128 columns
  static constexpr int ROUNDS = 32 * 32 / kTpThreads;   // 4: groups per thread in the row pass
};

// Element k (0..31) of a column gathered as 32 fp32 bit patterns.
template <int DT>
__device__ __forceinline__ void load_column(const uint4* tile, int c, uint32_t (&b)[32]) {
  constexpr int TILE_C = TileGeom<DT>::TILE_C;
  if (DT == FP8Q_BF16) {
    const uint16_t* t16 = reinterpret_cast<const uint16_t*>(tile);
#pragma unroll
    for (int r = 0; r < 32; ++r) b[r] = (uint32_t)t16[r * TILE_C + c] << 16;
  } else {
    const uint32_t* t32 = reinterpret_cast<const uint32_t*>(tile);
#pragma unroll
    for (int r = 0; r < 32; ++r) b[r] = t32[r * TILE_C + c];
  }
}

// Cast 32 values (fp32 bits) with scale s into 32 bytes.
template <int FMT>
__device__ __forceinline__ void cast32(const uint32_t (&b)[32], float s, uint32_t (&o)[8]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t lo = cvt_pair<FMT>(__uint_as_float(b[4 * k]) * s, __uint_as_float(b[4 * k + 1]) * s);
    const uint32_t hi = cvt_pair<FMT>(__uint_as_float(b[4 * k + 2]) * s, __uint_as_float(b[4 * k + 3]) * s);
    o[k] = lo | (hi << 16);
  }
}

__device__ __forceinline__ void set_byte(uint32_t (&o)[8], int k, uint32_t byte) {
  const int sh = (k & 3) * 8;
  o[k >> 2] = (o[k >> 2] & ~(0xFFu << sh)) | (byte << sh);
}

__device__ __forceinline__ void store32(uint8_t* dst, const uint32_t (&o)[8]) {
  __stcs(reinterpret_cast<uint4*>(dst), make_uint4(o[0], o[1], o[2], o[3]));
  __stcs(reinterpret_cast<uint4*>(dst) + 1, make_uint4(o[4], o[5], o[6], o[7]));
}

// bf16 column pairs: a 32-bit shared word holds columns 2p (low half) and
// 2p + 1 (high half) of one row, so a pair costs one load per row.
template <int HI>
__device__ __forceinline__ uint32_t half_bits(uint32_t w) {
  return HI ? (w & 0xFFFF0000u) : (w << 16);
}

template <int FMT, int HI>
__device__ __forceinline__ void cast32_half(const uint32_t (&w)[32], float s, uint32_t (&o)[8]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t lo = cvt_pair<FMT>(__uint_as_float(half_bits<HI>(w[4 * k])) * s,
                                      __uint_as_float(half_bits<HI>(w[4 * k + 1])) * s);
    const uint32_t hi = cvt_pair<FMT>(__uint_as_float(half_bits<HI>(w[4 * k + 2])) * s,
                                      __uint_as_float(half_bits<HI>(w[4 * k + 3])) * s);
    o[k] = lo | (hi << 16);
  }
}

__device__ __forceinline__ void load_pair_column(const uint4* tile, int p, uint32_t (&w)[32]) {
  const uint32_t* t32 = reinterpret_cast<const uint32_t*>(tile);
#pragma unroll
  for (int r = 0; r < 32; ++r) w[r] = t32[r * 128 + p];
}

// One MX column block (half HI of a bf16 column pair): E8M0 byte, 32 bytes.
template <int FMT, int HI>
__device__ __forceinline__ void mx_column_half(const uint32_t (&w)[32], uint32_t m, int rule, int headroom,
                                               uint32_t& clip, uint8_t* dst, uint8_t* e8dst) {
  uint32_t o[8];
  uint32_t ebyte;
  if (m >= 0x7F800000u) {
    ebyte = 0xFFu;
#pragma unroll
    for (int k = 0; k < 32; ++k) set_byte(o, k, ((half_bits<HI>(w[k]) >> 31) << 7) | 0x7Fu);
  } else {
    const int E = block_exp<FMT>(m, rule, headroom);
    ebyte = (uint32_t)(E + 127);
    const float s = __uint_as_float((uint32_t)(127 - E) << 23);
    cast32_half<FMT, HI>(w, s, o);
    const int be = (int)(fmax_bits(FMT) >> 23) + E;
    if (be < 255 && m > fmax_bits(FMT) + ((uint32_t)E << 23)) {
#pragma unroll
      for (int k = 0; k < 32; ++k) clip += clips<FMT>(__uint_as_float(half_bits<HI>(w[k])) * s) ? 1u : 0u;
    }
  }
  store32(dst, o);
  *e8dst = (uint8_t)ebyte;
}

// One per-tensor column (half HI of a bf16 column pair) with scale s.
template <int FMT, int HI>
__device__ __forceinline__ void ct_column_half(const uint32_t (&w)[32], uint32_t m, float s, uint8_t* dst) {
  uint32_t o[8];
  cast32_half<FMT, HI>(w, s, o);
  if (m > 0x7F800000u) {                                 // a NaN in the column
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const uint32_t b = half_bits<HI>(w[k]);
      if ((b & 0x7FFFFFFFu) > 0x7F800000u) set_byte(o, k, ((b >> 31) << 7) | 0x7Fu);
    }
  }
  store32(dst, o);
}

// Shared pipeline bookkeeping of both kernels: this CTA's tiles are
// blockIdx.x + j * gridDim.x; thread 0 keeps kTpStages - 1 tiles in flight.
struct TilePipe {
  const CUtensorMap* map;
  uint4* stages;
  uint64_t* full;
  int64_t col_tiles, mine;
  int tile_c;

  __device__ __forceinline__ void issue(int64_t j) const {
    const int64_t t = blockIdx.x + j * (int64_t)gridDim.x;
    const int st = (int)(j % kTpStages);
    mbar_arrive_expect_tx(&full[st], kTpTileBytes);
    tma_load_2d(stages + st * (kTpTileBytes / 16), map, &full[st], (int)((t % col_tiles) * tile_c),
                (int)((t / col_tiles) * 32));
  }
  __device__ __forceinline__ void start() const {
    if (threadIdx.x == 0) {
      for (int i = 0; i < kTpStages; ++i) mbar_init(&full[i], 1);
      fence_barrier_init();
      prefetch_tensormap(map);
    }
    __syncthreads();
    if (threadIdx.x == 0)
      for (int64_t j = 0; j < kTpStages - 1 && j < mine; ++j) issue(j);
  }
  // Refill, then wait for tile j.  False (for every thread) when some thread's
  // wait ran out of time: the caller then stops.
  __device__ __forceinline__ bool next(int64_t j) const {
    if (threadIdx.x == 0 && j + kTpStages - 1 < mine) {
      fence_proxy_async();
      issue(j + kTpStages - 1);
    }
    const bool ok = mbar_wait(&full[j % kTpStages], (uint32_t)((j / kTpStages) & 1));
    if (__syncthreads_or(!ok)) {
      if (threadIdx.x == 0) {
        note_wait_timeout();
        for (int64_t k = j; k < j + kTpStages - 1 && k < mine; ++k)   // bounded drain
          mbar_wait(&full[k % kTpStages], (uint32_t)((k / kTpStages) & 1));
      }
      return false;
    }
    return true;
  }
  __device__ __forceinline__ const uint4* tile(int64_t j) const {
    return stages + (j % kTpStages) * (kTpTileBytes / 16);
  }
};

__device__ __forceinline__ uint4* aligned_stages(uint4* dyn) {
  return reinterpret_cast<uint4*>(reinterpret_cast<char*>(dyn) +
                                  ((1024u - (smem_addr(dyn) & 1023u)) & 1023u));
}

// ---------------------------------------------------------------------------
// MX dual cast
// ---------------------------------------------------------------------------

template <int DT, int FMT>
__global__ void __launch_bounds__(kTpThreads, 2) mx_dual_kernel(
    const __grid_constant__ CUtensorMap tmap, int64_t rows, int64_t cols, int rule, int headroom,
    uint8_t* __restrict__ q_row, uint8_t* __restrict__ e8_row, uint8_t* __restrict__ q_colt,
    uint8_t* __restrict__ e8_colt, unsigned long long* clipped_row, unsigned long long* clipped_col) {
  using G = TileGeom<DT>;
  constexpr int EPL = G::EPL, TILE_C = G::TILE_C;
  constexpr int LPB = 32 / EPL;                      // lanes per row block in the row pass
  extern __shared__ __align__(1024) uint4 dyn_smem[];
  __shared__ __align__(8) uint64_t full[kTpStages];
  __shared__ uint32_t red[2][kTpThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  TilePipe pipe;
  pipe.map = &tmap;
  pipe.stages = aligned_stages(dyn_smem);
  pipe.full = full;
  pipe.tile_c = TILE_C;
  pipe.col_tiles = (cols + TILE_C - 1) / TILE_C;
  const int64_t ntiles = (rows / 32) * pipe.col_tiles;
  pipe.mine = ntiles > (int64_t)blockIdx.x ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  pipe.start();
  const int64_t cb = cols / 32, rb = rows / 32;      // e8m0 row lengths
  uint32_t clip_r = 0, clip_c = 0;
  for (int64_t j = 0; j < pipe.mine; ++j) {
    if (!pipe.next(j)) return;
    const uint4* tile = pipe.tile(j);
    const int64_t t = blockIdx.x + j * (int64_t)gridDim.x;
    const int64_t r0 = (t / pipe.col_tiles) * 32, c0 = (t % pipe.col_tiles) * TILE_C;

    // A. row-wise blocks
#pragma unroll
    for (int i = 0; i < G::ROUNDS; ++i) {
      const int r = warp * G::ROUNDS + i;            // tile row; lane = 16-byte group
      const uint4 v = tile[r * 32 + lane];
      uint32_t m = unpack_max<DT>(absmax_load<DT>(v));
#pragma unroll
      for (int o = 1; o < LPB; o <<= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      const int64_t col = c0 + (int64_t)lane * EPL;
      uint2 out;
      uint32_t ebyte;
      if (m >= 0x7F800000u) {                        // NaN / Inf block
        ebyte = 0xFFu;
        uint32_t w[2] = {0u, 0u};
#pragma unroll
        for (int k = 0; k < EPL; ++k) w[k >> 2] |= ((((elem_bits<DT>(v, k) >> 31) << 7) | 0x7Fu) << ((k & 3) * 8));
        out = make_uint2(w[0], w[1]);
      } else {
        const int E = block_exp<FMT>(m, rule, headroom);
        ebyte = (uint32_t)(E + 127);
        const float s = __uint_as_float((uint32_t)(127 - E) << 23);
        out = cast_load<DT, FMT>(v, s);
        const int be = (int)(fmax_bits(FMT) >> 23) + E;
        if (be < 255 && m > fmax_bits(FMT) + ((uint32_t)E << 23)) {
#pragma unroll
          for (int k = 0; k < EPL; ++k) clip_r += clips<FMT>(__uint_as_float(elem_bits<DT>(v, k)) * s) ? 1u : 0u;
        }
      }
      if (col < cols) {
        uint8_t* dst = q_row + (r0 + r) * cols + col;
        if (DT == FP8Q_BF16) __stcs(reinterpret_cast<uint2*>(dst), out);
        else __stcs(reinterpret_cast<unsigned int*>(dst), out.x);
        if ((lane & (LPB - 1)) == 0) e8_row[(r0 + r) * cb + (col >> 5)] = (uint8_t)ebyte;
      }
    }

    // B. column-wise blocks, written transposed
    if (DT == FP8Q_BF16) {
      if (tid < TILE_C / 2 && c0 + 2 * tid < cols) {      // one bf16 column pair per thread
        uint32_t w[32];
        load_pair_column(tile, tid, w);
        uint32_t pm = 0;
#pragma unroll
        for (int k = 0; k < 32; ++k) pm = vmax_u16x2(pm, w[k] & 0x7FFF7FFFu);
        const int64_t c = c0 + 2 * tid;
        mx_column_half<FMT, 0>(w, pm << 16, rule, headroom, clip_c, q_colt + c * rows + r0,
                               e8_colt + c * rb + (r0 >> 5));
        mx_column_half<FMT, 1>(w, pm & 0xFFFF0000u, rule, headroom, clip_c,
                               q_colt + (c + 1) * rows + r0, e8_colt + (c + 1) * rb + (r0 >> 5));
      }
    } else if (tid < TILE_C && c0 + tid < cols) {
      uint32_t b[32];
      load_column<DT>(tile, tid, b);
      uint32_t m = 0;
#pragma unroll
      for (int k = 0; k < 32; ++k) m = max(m, b[k] & 0x7FFFFFFFu);
      uint32_t o[8];
      uint32_t ebyte;
      if (m >= 0x7F800000u) {
        ebyte = 0xFFu;
#pragma unroll
        for (int k = 0; k < 32; ++k) set_byte(o, k, ((b[k] >> 31) << 7) | 0x7Fu);
      } else {
        const int E = block_exp<FMT>(m, rule, headroom);
        ebyte = (uint32_t)(E + 127);
        const float s = __uint_as_float((uint32_t)(127 - E) << 23);
        cast32<FMT>(b, s, o);
        const int be = (int)(fmax_bits(FMT) >> 23) + E;
        if (be < 255 && m > fmax_bits(FMT) + ((uint32_t)E << 23)) {
#pragma unroll
          for (int k = 0; k < 32; ++k) clip_c += clips<FMT>(__uint_as_float(b[k]) * s) ? 1u : 0u;
        }
      }
      const int64_t c = c0 + tid;
      store32(q_colt + c * rows + r0, o);
      e8_colt[c * rb + (r0 >> 5)] = (uint8_t)ebyte;
    }
    __syncthreads();                                 // the stage is free for the refill
  }
  clip_r = __reduce_add_sync(0xFFFFFFFFu, clip_r);
  clip_c = __reduce_add_sync(0xFFFFFFFFu, clip_c);
  if (lane == 0) { red[0][warp] = clip_r; red[1][warp] = clip_c; }
  __syncthreads();
  if (tid == 0) {
    unsigned long long a = 0, b = 0;
    for (int i = 0; i < kTpThreads / 32; ++i) { a += red[0][i]; b += red[1][i]; }
    if (clipped_row && a) atomicAdd(clipped_row, a);
    if (clipped_col && b) atomicAdd(clipped_col, b);
  }
}

// ---------------------------------------------------------------------------
// Per-tensor cast + transpose
// ---------------------------------------------------------------------------

template <int DT, int FMT>
__global__ void __launch_bounds__(kTpThreads, 2) cast_transpose_kernel(
    const __grid_constant__ CUtensorMap tmap, int64_t rows, int64_t cols, uint8_t* __restrict__ q,
    uint8_t* __restrict__ qt, DevState* st, int mode, GroupHeader h) {
  using G = TileGeom<DT>;
  constexpr int EPL = G::EPL, TILE_C = G::TILE_C;
  extern __shared__ __align__(1024) uint4 dyn_smem[];
  __shared__ __align__(8) uint64_t full[kTpStages];
  __shared__ int s_e;
  __shared__ uint32_t s_nonfin;
  __shared__ uint32_t red_m[kTpThreads / 32], red_c[kTpThreads / 32];
  const int tid = threadIdx.x;
  TilePipe pipe;
  pipe.map = &tmap;
  pipe.stages = aligned_stages(dyn_smem);
  pipe.full = full;
  pipe.tile_c = TILE_C;
  pipe.col_tiles = (cols + TILE_C - 1) / TILE_C;
  const int64_t ntiles = (rows / 32) * pipe.col_tiles;
  pipe.mine = ntiles > (int64_t)blockIdx.x ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  if (tid == 0) s_nonfin = 0u;
  if (tid < 32) warp_exp(st, mode, &s_e);
  pipe.start();                                      // its barrier publishes s_e and s_nonfin
  const int e = s_e;
  const float s = pow2f(e);
  const uint32_t bound = no_clip_bound(FMT, e);
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t lmax = 0, lclip = 0;
  for (int64_t j = 0; j < pipe.mine; ++j) {
    if (!pipe.next(j)) return;
    const uint4* tile = pipe.tile(j);
    const int64_t t = blockIdx.x + j * (int64_t)gridDim.x;
    const int64_t r0 = (t / pipe.col_tiles) * 32, c0 = (t % pipe.col_tiles) * TILE_C;
    // A. row-major: one 16-byte group per lane per round
#pragma unroll
    for (int i = 0; i < G::ROUNDS; ++i) {
      const int r = warp * G::ROUNDS + i;
      const uint4 v = tile[r * 32 + lane];
      const uint32_t m = unpack_max<DT>(absmax_load<DT>(v));
      lmax = max(lmax, m);
      uint2 out = cast_load<DT, FMT>(v, s);
      if (m > bound) fix_load<DT, FMT>(v, s, out, lclip, &s_nonfin);
      const int64_t col = c0 + (int64_t)lane * EPL;
      if (col < cols) {
        uint8_t* dst = q + (r0 + r) * cols + col;
        if (DT == FP8Q_BF16) __stcs(reinterpret_cast<uint2*>(dst), out);
        else __stcs(reinterpret_cast<unsigned int*>(dst), out.x);
      }
    }
    // B. transposed (clipping was counted in A)
    if (DT == FP8Q_BF16) {
      if (tid < TILE_C / 2 && c0 + 2 * tid < cols) {      // one bf16 column pair per thread
        uint32_t w[32];
        load_pair_column(tile, tid, w);
        uint32_t pm = 0;
#pragma unroll
        for (int k = 0; k < 32; ++k) pm = vmax_u16x2(pm, w[k] & 0x7FFF7FFFu);
        const int64_t c = c0 + 2 * tid;
        ct_column_half<FMT, 0>(w, pm << 16, s, qt + c * rows + r0);
        ct_column_half<FMT, 1>(w, pm & 0xFFFF0000u, s, qt + (c + 1) * rows + r0);
      }
    } else if (tid < TILE_C && c0 + tid < cols) {
      uint32_t b[32];
      load_column<DT>(tile, tid, b);
      uint32_t o[8];
      cast32<FMT>(b, s, o);
      uint32_t m = 0;
#pragma unroll
      for (int k = 0; k < 32; ++k) m = max(m, b[k] & 0x7FFFFFFFu);
      if (m > 0x7F800000u) {                          // a NaN in the column
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if ((b[k] & 0x7FFFFFFFu) > 0x7F800000u) set_byte(o, k, ((b[k] >> 31) << 7) | 0x7Fu);
      }
      store32(qt + (c0 + tid) * rows + r0, o);
    }
    __syncthreads();
  }
  // per-CTA totals, then the ticket: the CTA completing the tensor finishes it
  uint32_t cnt = lclip;
  lmax = __reduce_max_sync(0xFFFFFFFFu, lmax);
  cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
  if (lane == 0) { red_m[warp] = lmax; red_c[warp] = cnt; }
  __syncthreads();
  if (tid == 0 && pipe.mine > 0) {
    for (int i = 1; i < kTpThreads / 32; ++i) { lmax = max(lmax, red_m[i]); cnt += red_c[i]; }
    if (lmax) atomicMax(&st->amax_acc, lmax);
    if (cnt) atomicAdd(&st->clip_acc, (unsigned long long)cnt);
    if (s_nonfin) atomicAdd(&st->nonfinite_acc, (unsigned long long)s_nonfin);
    __threadfence();
    const unsigned done = (unsigned)pipe.mine;
    const unsigned prev = atomicAdd(&st->ticket, done);
    if (prev + done == (unsigned)ntiles) finish_tensor(st, h, 0, e);
  }
}

// ---------------------------------------------------------------------------
// launches
// ---------------------------------------------------------------------------

template <int DT, int FMT>
static cudaError_t launch_dual_t(const void* x, int64_t rows, int64_t cols, int rule, int headroom,
                                 uint8_t* q_row, uint8_t* e8_row, uint8_t* q_colt, uint8_t* e8_colt,
                                 unsigned long long* cr, unsigned long long* cc, cudaStream_t s,
                                 int* launches) {
  constexpr int TILE_C = TileGeom<DT>::TILE_C;
  auto kern = mx_dual_kernel<DT, FMT>;
  int occ = 1;
  cudaError_t e = kernel_occupancy(reinterpret_cast<const void*>(kern), kTpThreads,
                                   kTpStages * kTpTileBytes + 1024, &occ);
  if (e != cudaSuccess) return e;
  CUtensorMap map;
  e = encode_tile_map(&map, x, DT == FP8Q_BF16, rows, cols, TILE_C);
  if (e != cudaSuccess) return e;
  const int64_t ntiles = (rows / 32) * ((cols + TILE_C - 1) / TILE_C);
  long long grid = (long long)sm_count(device_of_current()) * occ;
  if (grid > ntiles) grid = ntiles;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, kTpThreads, kTpStages * kTpTileBytes + 1024, s>>>(map, rows, cols, rule, headroom, q_row,
                                                                          e8_row, q_colt, e8_colt, cr, cc);
  ++*launches;
  return cudaGetLastError();
}

cudaError_t launch_mx_dual(const void* x, int dtype, int64_t rows, int64_t cols, int format, int rule,
                           int headroom, uint8_t* q_row, uint8_t* e8_row, uint8_t* q_colt,
                           uint8_t* e8_colt, unsigned long long* cr, unsigned long long* cc,
                           cudaStream_t s, int* launches) {
  if (dtype == FP8Q_BF16)
    return format == FP8Q_E4M3
               ? launch_dual_t<FP8Q_BF16, FP8Q_E4M3>(x, rows, cols, rule, headroom, q_row, e8_row, q_colt, e8_colt, cr, cc, s, launches)
               : launch_dual_t<FP8Q_BF16, FP8Q_E5M2>(x, rows, cols, rule, headroom, q_row, e8_row, q_colt, e8_colt, cr, cc, s, launches);
  return format == FP8Q_E4M3
             ? launch_dual_t<FP8Q_F32, FP8Q_E4M3>(x, rows, cols, rule, headroom, q_row, e8_row, q_colt, e8_colt, cr, cc, s, launches)
             : launch_dual_t<FP8Q_F32, FP8Q_E5M2>(x, rows, cols, rule, headroom, q_row, e8_row, q_colt, e8_colt, cr, cc, s, launches);
}

template <int DT, int FMT>
static cudaError_t launch_ct_t(const void* x, int64_t rows, int64_t cols, uint8_t* q, uint8_t* qt,
                               DevState* st, int mode, const GroupHeader& h, cudaStream_t s,
                               int* launches) {
  constexpr int TILE_C = TileGeom<DT>::TILE_C;
  auto kern = cast_transpose_kernel<DT, FMT>;
  int occ = 1;
  cudaError_t e = kernel_occupancy(reinterpret_cast<const void*>(kern), kTpThreads,
                                   kTpStages * kTpTileBytes + 1024, &occ);
  if (e != cudaSuccess) return e;
  CUtensorMap map;
  e = encode_tile_map(&map, x, DT == FP8Q_BF16, rows, cols, TILE_C);
  if (e != cudaSuccess) return e;
  const int64_t ntiles = (rows / 32) * ((cols + TILE_C - 1) / TILE_C);
  long long grid = (long long)sm_count(device_of_current()) * occ;
  if (grid > ntiles) grid = ntiles;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, kTpThreads, kTpStages * kTpTileBytes + 1024, s>>>(map, rows, cols, q, qt, st, mode, h);
  ++*launches;
  return cudaGetLastError();
}

cudaError_t launch_cast_transpose(const void* x, int dtype, int format, int64_t rows, int64_t cols,
                                  uint8_t* q, uint8_t* qt, DevState* st, int mode, const GroupHeader& h,
                                  cudaStream_t s, int* launches) {
  if (dtype == FP8Q_BF16)
    return format == FP8Q_E4M3 ? launch_ct_t<FP8Q_BF16, FP8Q_E4M3>(x, rows, cols, q, qt, st, mode, h, s, launches)
                               : launch_ct_t<FP8Q_BF16, FP8Q_E5M2>(x, rows, cols, q, qt, st, mode, h, s, launches);
  return format == FP8Q_E4M3 ? launch_ct_t<FP8Q_F32, FP8Q_E4M3>(x, rows, cols, q, qt, st, mode, h, s, launches)
                             : launch_ct_t<FP8Q_F32, FP8Q_E5M2>(x, rows, cols, q, qt, st, mode, h, s, launches);
}

}  // namespace fp8q

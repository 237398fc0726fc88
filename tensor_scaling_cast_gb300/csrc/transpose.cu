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
// Every warp runs its own pipeline: it streams 32-row x 128-byte sub-tiles
// (64 bf16 / 32 fp32 columns, 4 KiB) through a few shared-memory stages
// filled by cp.async.bulk.tensor.2d with the 128-byte swizzle, one mbarrier
// per stage and bounded waits.  Warps never wait for one another.  Lane l of
// a warp owns, per sub-tile:
//   A. row pass: row l, i.e. 2 (bf16) / 1 (fp32) 32-element row blocks, read
//      as 16-byte chunks and written as 32 contiguous bytes each;
//   B. column pass: bf16 columns 2l and 2l + 1 (one 32-bit word per row) or
//      fp32 column l, written as 32 contiguous bytes of the transposed
//      output per column.
// The swizzle puts chunk c of tile row r at chunk c ^ (r & 7), so both the
// row pass (8 rows per quarter-warp, same logical chunk) and the column pass
// (32 words of one row) touch 32 distinct banks.
#include <cuda.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "fp8q_device.cuh"
#include "fp8q_internal.cuh"
#include "state.cuh"
#include "tma.cuh"

namespace fp8q {

// Pipeline shape of each kernel (input stages per warp, output staging
// buffers per warp, row tiles per chunk), overridable at build time.
#ifndef FP8Q_DUAL_STAGES
#define FP8Q_DUAL_STAGES 2
#endif
#ifndef FP8Q_DUAL_OBUF
#define FP8Q_DUAL_OBUF 2
#endif
#ifndef FP8Q_DUAL_CHUNK
#define FP8Q_DUAL_CHUNK 4
#endif
#ifndef FP8Q_CT_STAGES
#define FP8Q_CT_STAGES 2
#endif
#ifndef FP8Q_CT_OBUF
#define FP8Q_CT_OBUF 2
#endif
#ifndef FP8Q_CT_CHUNK
#define FP8Q_CT_CHUNK 1
#endif
#ifndef FP8Q_DUAL_COLF
#define FP8Q_DUAL_COLF true
#endif
#ifndef FP8Q_CT_COLF
#define FP8Q_CT_COLF false
#endif
#ifndef FP8Q_TP_L2PROMO
#define FP8Q_TP_L2PROMO 128
#endif
#ifndef FP8Q_TP_MINB
#define FP8Q_TP_MINB 4
#endif
constexpr int kWWarps = 4;                             // warps per CTA
constexpr int kWThreads = 32 * kWWarps;
constexpr int kWTileBytes = 32 * 128;                  // 32 rows x 128 bytes
constexpr int kWTileVec = kWTileBytes / 16;            // uint4 per sub-tile
constexpr int kWOutBytes = 2 * 2048;                   // staging: row-major part + transposed part

template <int S, int OB, int CH, bool COLF>
struct TpCfg {
  static_assert(S >= 2 && S <= 8, "input stages");
  static_assert(OB == 1 || OB == 2, "one or two output staging buffers");
  static_assert(CH >= 1 && CH <= 8, "the column E8M0 run is kept in one 64-bit word");
  static constexpr int kStages = S, kOutBufs = OB, kChunk = CH;
  static constexpr bool kColFastest = COLF;      // chunk order: column tile fastest
  static constexpr int kWarpBytes = S * kWTileBytes + OB * kWOutBytes;
  static constexpr int kSmemBytes = kWWarps * kWarpBytes + 1024;   // + alignment slack
};
using DualCfg = TpCfg<FP8Q_DUAL_STAGES, FP8Q_DUAL_OBUF, FP8Q_DUAL_CHUNK, FP8Q_DUAL_COLF>;
using CtCfg = TpCfg<FP8Q_CT_STAGES, FP8Q_CT_OBUF, FP8Q_CT_CHUNK, FP8Q_CT_COLF>;

static __device__ unsigned int g_tp_wait_timeouts;   // see fp8q_pipeline_status

__device__ __forceinline__ void note_wait_timeout() { atomicAdd(&g_tp_wait_timeouts, 1u); }

cudaError_t read_tp_wait_timeouts(unsigned int* count) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(count, g_tp_wait_timeouts, sizeof(unsigned int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_tp_wait_timeouts, &zero, sizeof(unsigned int));
  return e;
}

template <int DT>
struct TileGeom {
  static constexpr int EPL = DT == FP8Q_BF16 ? 8 : 4;   // elements per 16-byte group
  static constexpr int TILE_C = 8 * EPL;                // 64 / 32 columns per sub-tile
  static constexpr int NG = 32 / EPL;                   // 16-byte chunks per 32-element block
  static constexpr int BPR = TILE_C / 32;               // row blocks per sub-tile row
};

// The 32 bytes of a row block from its NG per-chunk casts.
template <int DT, int NG>
__device__ __forceinline__ void pack_row(const uint2 (&t)[NG], uint32_t (&o)[8]) {
#pragma unroll
  for (int k = 0; k < NG; ++k) {
    if (DT == FP8Q_BF16) {
      o[2 * k] = t[k].x;
      o[2 * k + 1] = t[k].y;
    } else {
      o[k] = t[k].x;
    }
  }
}

// Max of |.| over 32 words as a depth-5 tree (a serial chain would leave
// each thread waiting on 32 dependent max operations).  Packed bf16 pairs
// (PAIRS) or fp32 bit patterns.
template <bool PAIRS>
__device__ __forceinline__ uint32_t tree_absmax32(const uint32_t (&w)[32]) {
  const uint32_t mask = PAIRS ? 0x7FFF7FFFu : 0x7FFFFFFFu;
  uint32_t t[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    t[i] = PAIRS ? vmax_u16x2(w[2 * i] & mask, w[2 * i + 1] & mask) : max(w[2 * i] & mask, w[2 * i + 1] & mask);
#pragma unroll
  for (int n = 8; n >= 1; n >>= 1)
#pragma unroll
    for (int i = 0; i < n; ++i) t[i] = PAIRS ? vmax_u16x2(t[2 * i], t[2 * i + 1]) : max(t[2 * i], t[2 * i + 1]);
  return t[0];
}

// Word l of each of the 32 rows of a swizzled sub-tile: a bf16 column pair
// (column 2l in the low half, 2l + 1 in the high half) or fp32 column l.
__device__ __forceinline__ void load_column_words(const uint4* tile, int l, uint32_t (&w)[32]) {
  const uint32_t* t32 = reinterpret_cast<const uint32_t*>(tile);
#pragma unroll
  for (int r = 0; r < 32; ++r) w[r] = t32[r * 32 + (l ^ ((r & 7) << 2))];
}

// The NG 16-byte chunks of row block b of swizzled tile row r.
template <int NG>
__device__ __forceinline__ void load_row_block(const uint4* tile, int r, int b, uint4 (&v)[NG]) {
#pragma unroll
  for (int k = 0; k < NG; ++k) v[k] = tile[r * 8 + ((b * NG + k) ^ (r & 7))];
}

// fp32 bits of element k of a column: half HI of the word for bf16 pairs,
// the whole word for fp32 (HI = 2).
template <int HI>
__device__ __forceinline__ uint32_t half_bits(uint32_t w) {
  return HI == 2 ? w : HI ? (w & 0xFFFF0000u) : (w << 16);
}

// Cast the 32 values of a column with scale s into 32 bytes.
template <int FMT, int HI>
__device__ __forceinline__ void cast32(const uint32_t (&w)[32], float s, uint32_t (&o)[8]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t lo = cvt_pair<FMT>(__uint_as_float(half_bits<HI>(w[4 * k])) * s,
                                      __uint_as_float(half_bits<HI>(w[4 * k + 1])) * s);
    const uint32_t hi = cvt_pair<FMT>(__uint_as_float(half_bits<HI>(w[4 * k + 2])) * s,
                                      __uint_as_float(half_bits<HI>(w[4 * k + 3])) * s);
    o[k] = lo | (hi << 16);
  }
}

__device__ __forceinline__ void set_byte(uint32_t (&o)[8], int k, uint32_t byte) {
  const int sh = (k & 3) * 8;
  o[k >> 2] = (o[k >> 2] & ~(0xFFu << sh)) | (byte << sh);
}

// Output staging.  Each warp writes the 8-bit outputs of a sub-tile into a
// shared-memory buffer that a TMA tiled store then copies out: the
// row-major part (32 rows x TILE_C bytes) at offset 0 and the transposed part
// (TILE_C rows x 32 bytes) at offset 2048, both in the swizzled layout of
// their tensor maps (64-byte rows: chunk c of row r at c ^ ((r >> 1) & 3);
// 32-byte rows: chunk c of row r at c ^ ((r >> 2) & 1)), which keeps the
// warp's 16-byte shared stores free of bank conflicts (the transposed part of
// a bf16 sub-tile: two-way).
template <int ROWB>
__device__ __forceinline__ void stage16(uint8_t* buf, int r, int c, uint32_t a, uint32_t b, uint32_t cc,
                                        uint32_t d) {
  const int sw = ROWB == 64 ? ((r >> 1) & 3) : ((r >> 2) & 1);
  *reinterpret_cast<uint4*>(buf + r * ROWB + ((c ^ sw) << 4)) = make_uint4(a, b, cc, d);
}
// 32 bytes o into row r at byte offset 32 * half of a staging part with
// ROWB-byte rows.
template <int ROWB>
__device__ __forceinline__ void stage32(uint8_t* buf, int r, int half, const uint32_t (&o)[8]) {
  stage16<ROWB>(buf, r, 2 * half, o[0], o[1], o[2], o[3]);
  stage16<ROWB>(buf, r, 2 * half + 1, o[4], o[5], o[6], o[7]);
}

// One MX column block (column HI of the lane's words): its 32 bytes into o,
// returns its E8M0 byte.  m = the block's max |x| bits.
template <int FMT, int HI>
__device__ __forceinline__ uint32_t mx_column(const uint32_t (&w)[32], uint32_t m, int rule, int headroom,
                                              uint32_t& clip, uint32_t (&o)[8]) {
  uint32_t ebyte;
  if (m >= 0x7F800000u) {                              // NaN / Inf block
    ebyte = 0xFFu;
#pragma unroll
    for (int k = 0; k < 32; ++k) set_byte(o, k, ((half_bits<HI>(w[k]) >> 31) << 7) | 0x7Fu);
  } else {
    const int E = block_exp<FMT>(m, rule, headroom);
    ebyte = (uint32_t)(E + 127);
    const float s = __uint_as_float((uint32_t)(127 - E) << 23);
    cast32<FMT, HI>(w, s, o);
    const int be = (int)(fmax_bits(FMT) >> 23) + E;
    if (be < 255 && m > fmax_bits(FMT) + ((uint32_t)E << 23)) {
#pragma unroll
      for (int k = 0; k < 32; ++k) clip += clips<FMT>(__uint_as_float(half_bits<HI>(w[k])) * s) ? 1u : 0u;
    }
  }
  return ebyte;
}

// The E8M0 bytes of one column for the row tiles i0 .. i0 + n - 1 of a chunk
// (byte k of acc for row tile i0 + k), at e8 = the byte of row tile i0.  A
// full chunk at an address aligned to its size goes out as one store.
template <int CH>
using E8Acc = typename std::conditional<(CH > 4), unsigned long long, uint32_t>::type;
template <int CH>
__device__ __forceinline__ void store_e8_run(uint8_t* e8, E8Acc<CH> acc, uint32_t n) {
  if (n == (uint32_t)CH && (CH == 4 || CH == 8) && (reinterpret_cast<uintptr_t>(e8) & (CH - 1)) == 0) {
    *reinterpret_cast<E8Acc<CH>*>(e8) = acc;
    return;
  }
  for (uint32_t k = 0; k < n; ++k) e8[k] = (uint8_t)(acc >> (8 * k));
}

// One per-tensor column (column HI of the lane's words) with scale s.
// has_nan: the sub-tile holds a NaN somewhere (its sign must be kept).
template <int FMT, int HI>
__device__ __forceinline__ void ct_column(const uint32_t (&w)[32], bool has_nan, float s, uint32_t (&o)[8]) {
  cast32<FMT, HI>(w, s, o);
  if (has_nan) {
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const uint32_t b = half_bits<HI>(w[k]);
      if ((b & 0x7FFFFFFFu) > 0x7F800000u) set_byte(o, k, ((b >> 31) << 7) | 0x7Fu);
    }
  }
}

// Work order.  The sub-tiles form a grid of rtiles x ctiles (32 rows x
// tile_c columns each).  A chunk is CH consecutive row tiles of one
// column tile (fewer at the bottom edge); chunks are numbered row-chunk
// fastest and dealt to the warps round-robin (warp w takes chunks w,
// w + nwarps, ...).  Within a chunk a warp walks down the rows, so it can
// collect each column's CH transposed-scale bytes into one store.  The
// warps in flight together cover a band of adjacent column strips.
template <int CH, bool COLF>
struct TileCursor {
  uint32_t v;                    // chunk
  uint32_t fa, sl;               // its fast and slow coordinates
  uint32_t i;                    // row tile within the chunk
  __device__ __forceinline__ uint32_t rc() const { return COLF ? sl : fa; }
  __device__ __forceinline__ uint32_t ct() const { return COLF ? fa : sl; }
  __device__ __forceinline__ uint32_t rt() const { return rc() * CH + i; }
};

// One warp's pipeline over its chunks; lane 0 keeps up to C::kStages
// sub-tiles in flight.  Sub-tile counts are below 2^31 (checked by the
// launcher).
template <class C>
struct WarpPipe {
  static constexpr int kStages = C::kStages, kChunkR = C::kChunk;
  static constexpr bool kColF = C::kColFastest;
  using Cursor = TileCursor<kChunkR, kColF>;
  const CUtensorMap* map;
  uint4* stages;                 // this warp's kStages x 4 KiB
  uint64_t* full;                // this warp's kStages barriers
  uint32_t rtiles, nfast, nchunks, stride, sq, sr;
  uint32_t issued;               // lane 0: sub-tiles issued so far
  int tile_c;
  Cursor cur;                    // the sub-tile being processed
  Cursor next;                   // lane 0: the next sub-tile to issue

  __device__ __forceinline__ void setup(const CUtensorMap* m, uint4* st, uint64_t* f, uint32_t row_tiles,
                                        uint32_t col_tiles, int tc) {
    map = m;
    stages = st;
    full = f;
    tile_c = tc;
    rtiles = row_tiles;
    const uint32_t rchunks = (row_tiles + kChunkR - 1) / kChunkR;
    nchunks = rchunks * col_tiles;
    nfast = kColF ? col_tiles : rchunks;
    stride = gridDim.x * kWWarps;
    sq = stride / nfast;
    sr = stride % nfast;
    cur.v = blockIdx.x * kWWarps + (threadIdx.x >> 5);
    cur.sl = cur.v / nfast;
    cur.fa = cur.v % nfast;
    cur.i = 0;
    next = cur;
    issued = 0;
  }
  __device__ __forceinline__ bool valid(const Cursor& c) const { return c.v < nchunks; }
  // Last row tile of its chunk?
  __device__ __forceinline__ bool chunk_end(const Cursor& c) const {
    return c.i + 1 == (uint32_t)kChunkR || c.rt() + 1 >= rtiles;
  }
  __device__ __forceinline__ void step(Cursor& c) const {
    if (!chunk_end(c)) {
      ++c.i;
      return;
    }
    c.i = 0;
    c.v += stride;
    c.fa += sr;
    c.sl += sq;
    if (c.fa >= nfast) {
      c.fa -= nfast;
      ++c.sl;
    }
  }
  __device__ __forceinline__ int64_t r0() const { return (int64_t)cur.rt() * 32; }
  __device__ __forceinline__ int64_t c0() const { return (int64_t)cur.ct() * tile_c; }
  __device__ __forceinline__ void issue() {
    const int st = (int)(issued % kStages);
    mbar_arrive_expect_tx(&full[st], kWTileBytes);
    tma_load_2d(stages + st * kWTileVec, map, &full[st], (int)(next.ct() * tile_c), (int)(next.rt() * 32));
    step(next);
    ++issued;
  }
  // Barrier set-up and the first loads.  Warp-collective.
  __device__ __forceinline__ void start() {
    if ((threadIdx.x & 31) == 0) {
      for (int i = 0; i < kStages; ++i) mbar_init(&full[i], 1);
      fence_barrier_init();
      prefetch_tensormap(map);
      while (issued < (uint32_t)kStages && valid(next)) issue();
    }
    __syncwarp();
  }
  // Wait for the warp's sub-tile j (the current one).  False (for every
  // lane) when some lane's wait ran out of time: the loads still in flight
  // are waited for (bounded) and the caller stops.  Warp-collective.
  __device__ __forceinline__ bool wait(uint32_t j) const {
    const bool ok = mbar_wait(&full[j % kStages], (j / kStages) & 1u);
    if (__any_sync(0xFFFFFFFFu, !ok)) {
      if ((threadIdx.x & 31) == 0) {
        note_wait_timeout();
        for (uint32_t k = j; k < issued; ++k)        // bounded drain
          mbar_wait(&full[k % kStages], (k / kStages) & 1u);
      }
      return false;
    }
    return true;
  }
  // The warp is done with the current sub-tile: refill its stage and move
  // on.  Warp-collective.
  __device__ __forceinline__ void release() {
    __syncwarp();
    if ((threadIdx.x & 31) == 0 && valid(next)) {
      fence_proxy_async();
      issue();
    }
    step(cur);
  }
  __device__ __forceinline__ const uint4* tile(uint32_t j) const {
    return stages + (j % kStages) * kWTileVec;
  }
};

__device__ __forceinline__ uint4* aligned_stages(uint4* dyn) {
  return reinterpret_cast<uint4*>(reinterpret_cast<char*>(dyn) +
                                  ((1024u - (smem_addr(dyn) & 1023u)) & 1023u));
}

// Shared-memory regions of warp `warp`: its input stages, then its output
// staging buffers.
template <class C>
__device__ __forceinline__ uint8_t* warp_region(uint4* dyn, int warp) {
  return reinterpret_cast<uint8_t*>(aligned_stages(dyn)) + warp * C::kWarpBytes;
}

// Output staging of one warp: buffer k (of C::kOutBufs) for the warp's
// sub-tiles j with j modulo C::kOutBufs = k.  Lane 0 issues and commits the stores, so it
// alone waits for them.
template <class C>
struct OutStage {
  static constexpr int kOutBufs = C::kOutBufs;
  uint8_t* base;
  __device__ __forceinline__ uint8_t* buf(uint32_t j) const { return base + (j % kOutBufs) * kWOutBytes; }
  // Before writing buffer j: the store that last read it has read it.
  // Warp-collective.
  __device__ __forceinline__ void acquire() const {
    if ((threadIdx.x & 31) == 0) {
      if (kOutBufs == 1) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      else asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
    }
    __syncwarp();
  }
  // Buffer j is written: copy its two parts out.  Warp-collective.
  __device__ __forceinline__ void publish(uint32_t j, const CUtensorMap* qmap, const CUtensorMap* qtmap, int64_t r0,
                                         int64_t c0) const {
    fence_proxy_async();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
      tma_store_2d(qmap, buf(j), (int)c0, (int)r0);
      tma_store_2d(qtmap, buf(j) + 2048, (int)r0, (int)c0);
      bulk_commit();
    }
  }
  // Before the warp leaves: its stores are complete.  Warp-collective.
  __device__ __forceinline__ void drain() const {
    if ((threadIdx.x & 31) == 0) bulk_wait_all();
    __syncwarp();
  }
};

// ---------------------------------------------------------------------------
// MX dual cast
// ---------------------------------------------------------------------------

template <int DT, int FMT, class C>
__global__ void __launch_bounds__(kWThreads, FP8Q_TP_MINB) mx_dual_kernel(
    const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap qmap,
    const __grid_constant__ CUtensorMap qtmap, int64_t rows, int64_t cols, int rule, int headroom,
    uint8_t* __restrict__ e8_row, uint8_t* __restrict__ e8_colt, unsigned long long* clipped_row,
    unsigned long long* clipped_col) {
  using G = TileGeom<DT>;
  constexpr int EPL = G::EPL, TILE_C = G::TILE_C, NG = G::NG;
  constexpr int QROWB = TILE_C;                      // bytes per row of the row-major part
  extern __shared__ __align__(1024) uint4 dyn_smem[];
  __shared__ __align__(8) uint64_t full[kWWarps][C::kStages];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t ctiles = (uint32_t)((cols + TILE_C - 1) / TILE_C);
  uint8_t* region = warp_region<C>(dyn_smem, warp);
  WarpPipe<C> pipe;
  pipe.setup(&tmap, reinterpret_cast<uint4*>(region), full[warp], (uint32_t)(rows / 32), ctiles, TILE_C);
  const OutStage<C> out{region + C::kStages * kWTileBytes};
  pipe.start();
  const int64_t cb = cols / 32, rb = rows / 32;      // e8m0 row lengths
  uint32_t clip_r = 0, clip_c = 0;
  E8Acc<C::kChunk> e8c0 = 0, e8c1 = 0;                          // this chunk's column E8M0 bytes so far
  for (uint32_t j = 0; pipe.valid(pipe.cur); ++j) {
    if (!pipe.wait(j)) {
      out.drain();
      return;
    }
    const uint4* tile = pipe.tile(j);
    const int64_t r0 = pipe.r0(), c0 = pipe.c0();
    out.acquire();
    uint8_t* ob = out.buf(j);

    // A. row-wise blocks of tile row `lane`
    uint32_t ebytes = 0;
#pragma unroll
    for (int b = 0; b < G::BPR; ++b) {
      uint4 v[NG];
      load_row_block<NG>(tile, lane, b, v);
      uint32_t pm = absmax_load<DT>(v[0]);
#pragma unroll
      for (int k = 1; k < NG; ++k) pm = absmax_merge<DT>(pm, absmax_load<DT>(v[k]));
      const uint32_t m = unpack_max<DT>(pm);
      uint32_t o[8];
      uint32_t ebyte;
      if (m >= 0x7F800000u) {                        // NaN / Inf block
        ebyte = 0xFFu;
#pragma unroll
        for (int k = 0; k < 32; ++k) set_byte(o, k, ((elem_bits<DT>(v[k / EPL], k % EPL) >> 31) << 7) | 0x7Fu);
      } else {
        const int E = block_exp<FMT>(m, rule, headroom);
        ebyte = (uint32_t)(E + 127);
        const float s = __uint_as_float((uint32_t)(127 - E) << 23);
        uint2 t[NG];
#pragma unroll
        for (int k = 0; k < NG; ++k) t[k] = cast_load<DT, FMT>(v[k], s);
        pack_row<DT, NG>(t, o);
        const int be = (int)(fmax_bits(FMT) >> 23) + E;
        if (be < 255 && m > fmax_bits(FMT) + ((uint32_t)E << 23)) {
#pragma unroll
          for (int k = 0; k < 32; ++k)
            clip_r += clips<FMT>(__uint_as_float(elem_bits<DT>(v[k / EPL], k % EPL)) * s) ? 1u : 0u;
        }
      }
      stage32<QROWB>(ob, lane, b, o);
      ebytes |= ebyte << (8 * b);
    }
    {
      // this row's E8M0 bytes, adjacent: one 16-bit store for a full bf16 sub-tile row
      uint8_t* e8 = e8_row + (r0 + lane) * cb + (c0 >> 5);
      if (G::BPR == 2 && c0 + 64 <= cols) {
        if ((reinterpret_cast<uintptr_t>(e8) & 1u) == 0) {
          *reinterpret_cast<uint16_t*>(e8) = (uint16_t)ebytes;
        } else {
          e8[0] = (uint8_t)ebytes;
          e8[1] = (uint8_t)(ebytes >> 8);
        }
      } else {
        e8[0] = (uint8_t)ebytes;
      }
    }

    // B. column-wise blocks, transposed; their E8M0 bytes are collected over
    // the chunk's row tiles
    const uint32_t ci = pipe.cur.i;
    const bool flush = pipe.chunk_end(pipe.cur);
    const int64_t rt0 = (r0 >> 5) - ci;               // the chunk's first row tile
    uint32_t w[32], o[8];
    if (DT == FP8Q_BF16) {
      const int64_t c = c0 + 2 * lane;
      if (c < cols) {
        load_column_words(tile, lane, w);
        const uint32_t pm = tree_absmax32<true>(w);
        e8c0 |= (E8Acc<C::kChunk>)mx_column<FMT, 0>(w, pm << 16, rule, headroom, clip_c, o) << (8 * ci);
        stage32<32>(ob + 2048, 2 * lane, 0, o);
        e8c1 |= (E8Acc<C::kChunk>)mx_column<FMT, 1>(w, pm & 0xFFFF0000u, rule, headroom, clip_c, o) << (8 * ci);
        stage32<32>(ob + 2048, 2 * lane + 1, 0, o);
        if (flush) {
          store_e8_run<C::kChunk>(e8_colt + c * rb + rt0, e8c0, ci + 1);
          store_e8_run<C::kChunk>(e8_colt + (c + 1) * rb + rt0, e8c1, ci + 1);
        }
      }
    } else {
      const int64_t c = c0 + lane;
      if (c < cols) {
        load_column_words(tile, lane, w);
        e8c0 |= (E8Acc<C::kChunk>)mx_column<FMT, 2>(w, tree_absmax32<false>(w), rule, headroom, clip_c, o) << (8 * ci);
        stage32<32>(ob + 2048, lane, 0, o);
        if (flush) store_e8_run<C::kChunk>(e8_colt + c * rb + rt0, e8c0, ci + 1);
      }
    }
    if (flush) e8c0 = e8c1 = 0;
    out.publish(j, &qmap, &qtmap, r0, c0);
    pipe.release();
  }
  out.drain();
  clip_r = __reduce_add_sync(0xFFFFFFFFu, clip_r);
  clip_c = __reduce_add_sync(0xFFFFFFFFu, clip_c);
  if (lane == 0) {
    if (clipped_row && clip_r) atomicAdd(clipped_row, (unsigned long long)clip_r);
    if (clipped_col && clip_c) atomicAdd(clipped_col, (unsigned long long)clip_c);
  }
}

// ---------------------------------------------------------------------------
// Per-tensor cast + transpose
// ---------------------------------------------------------------------------

template <int DT, int FMT, class C>
__global__ void __launch_bounds__(kWThreads, FP8Q_TP_MINB) cast_transpose_kernel(
    const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap qmap,
    const __grid_constant__ CUtensorMap qtmap, int64_t rows, int64_t cols, DevState* st, int mode,
    GroupHeader h) {
  using G = TileGeom<DT>;
  constexpr int TILE_C = G::TILE_C, NG = G::NG;
  constexpr int QROWB = TILE_C;
  extern __shared__ __align__(1024) uint4 dyn_smem[];
  __shared__ __align__(8) uint64_t full[kWWarps][C::kStages];
  __shared__ int s_e;
  __shared__ uint32_t s_nonfin[kWWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t ctiles = (uint32_t)((cols + TILE_C - 1) / TILE_C);
  const uint32_t ntiles = (uint32_t)(rows / 32) * ctiles;
  uint8_t* region = warp_region<C>(dyn_smem, warp);
  WarpPipe<C> pipe;
  pipe.setup(&tmap, reinterpret_cast<uint4*>(region), full[warp], (uint32_t)(rows / 32), ctiles, TILE_C);
  const OutStage<C> out{region + C::kStages * kWTileBytes};
  pipe.start();
  if (lane == 0) s_nonfin[warp] = 0u;
  if (warp == 0) warp_exp(st, mode, &s_e);
  __syncthreads();                                   // publishes s_e
  const int e = s_e;
  const float s = pow2f(e);
  const uint32_t bound = no_clip_bound(FMT, e);
  uint32_t lmax = 0, lclip = 0;
  uint32_t j = 0;                                    // sub-tiles done by this warp
  for (; pipe.valid(pipe.cur); ++j) {
    if (!pipe.wait(j)) {
      out.drain();
      return;
    }
    const uint4* tile = pipe.tile(j);
    const int64_t r0 = pipe.r0(), c0 = pipe.c0();
    out.acquire();
    uint8_t* ob = out.buf(j);
    // A. row-major, tile row `lane`; clipping and non-finite inputs are counted here
    uint32_t tmax = 0;
#pragma unroll
    for (int b = 0; b < G::BPR; ++b) {
      uint4 v[NG];
      load_row_block<NG>(tile, lane, b, v);
      uint32_t pm = absmax_load<DT>(v[0]);
#pragma unroll
      for (int k = 1; k < NG; ++k) pm = absmax_merge<DT>(pm, absmax_load<DT>(v[k]));
      const uint32_t m = unpack_max<DT>(pm);
      tmax = max(tmax, m);
      uint2 t[NG];
#pragma unroll
      for (int k = 0; k < NG; ++k) t[k] = cast_load<DT, FMT>(v[k], s);
      if (m > bound) {
#pragma unroll
        for (int k = 0; k < NG; ++k) fix_load<DT, FMT>(v[k], s, t[k], lclip, &s_nonfin[warp]);
      }
      uint32_t o[8];
      pack_row<DT, NG>(t, o);
      stage32<QROWB>(ob, lane, b, o);
    }
    // B. transposed (a NaN anywhere in the sub-tile sends the columns through
    // the sign-keeping fix)
    lmax = max(lmax, tmax);
    const bool has_nan = __any_sync(0xFFFFFFFFu, tmax > 0x7F800000u);
    uint32_t w[32], o[8];
    if (DT == FP8Q_BF16) {
      if (c0 + 2 * lane < cols) {
        load_column_words(tile, lane, w);
        ct_column<FMT, 0>(w, has_nan, s, o);
        stage32<32>(ob + 2048, 2 * lane, 0, o);
        ct_column<FMT, 1>(w, has_nan, s, o);
        stage32<32>(ob + 2048, 2 * lane + 1, 0, o);
      }
    } else {
      if (c0 + lane < cols) {
        load_column_words(tile, lane, w);
        ct_column<FMT, 2>(w, has_nan, s, o);
        stage32<32>(ob + 2048, lane, 0, o);
      }
    }
    out.publish(j, &qmap, &qtmap, r0, c0);
    pipe.release();
  }
  out.drain();
  // per-warp totals, then the ticket: the warp completing the tensor finishes it
  lmax = __reduce_max_sync(0xFFFFFFFFu, lmax);
  const uint32_t cnt = __reduce_add_sync(0xFFFFFFFFu, lclip);
  __syncwarp();                                      // the warp's s_nonfin additions are done
  if (lane == 0 && j > 0) {
    if (lmax) atomicMax(&st->amax_acc, lmax);
    if (cnt) atomicAdd(&st->clip_acc, (unsigned long long)cnt);
    const uint32_t nf = s_nonfin[warp];
    if (nf) atomicAdd(&st->nonfinite_acc, (unsigned long long)nf);
    __threadfence();
    const unsigned prev = atomicAdd(&st->ticket, j);
    if (prev + j == ntiles) finish_tensor(st, h, 0, e);
  }
}

// ---------------------------------------------------------------------------
// launches
// ---------------------------------------------------------------------------

// Grid: as many CTAs as fit on the device at once, but no more warps than
// chunks.
template <int DT, class C>
static cudaError_t tp_grid(const void* kern, int64_t rows, int64_t cols, long long* grid) {
  constexpr int TILE_C = TileGeom<DT>::TILE_C;
  const int64_t ctiles = (cols + TILE_C - 1) / TILE_C;
  if ((rows / 32) * ctiles >= (int64_t(1) << 31)) return cudaErrorInvalidValue;   // 32-bit tile counts
  const int64_t nchunks = ((rows / 32 + C::kChunk - 1) / C::kChunk) * ctiles;
  int occ = 1;
  cudaError_t e = kernel_occupancy(kern, kWThreads, C::kSmemBytes, &occ);
  if (e != cudaSuccess) return e;
  long long gr = (long long)sm_count(device_of_current()) * occ;
  const long long need = (nchunks + kWWarps - 1) / kWWarps;
  if (gr > need) gr = need;
  *grid = gr < 1 ? 1 : gr;
  return cudaSuccess;
}

// The input map (32 rows x 128 bytes, 128-byte swizzle) and the two output
// maps (row-major q [rows, cols] and transposed qt [cols, rows], 8-bit).
template <int DT>
static cudaError_t tp_maps(const void* x, int64_t rows, int64_t cols, uint8_t* q, uint8_t* qt, CUtensorMap* in,
                           CUtensorMap* qmap, CUtensorMap* qtmap) {
  constexpr int TILE_C = TileGeom<DT>::TILE_C;
  cudaError_t e = encode_tile_map(in, x, DT == FP8Q_BF16, rows, cols, TILE_C, true, FP8Q_TP_L2PROMO);
  if (e == cudaSuccess) e = encode_byte_map(qmap, q, rows, cols, TILE_C, 32, TILE_C);
  if (e == cudaSuccess) e = encode_byte_map(qtmap, qt, cols, rows, 32, TILE_C, 32);
  return e;
}

template <int DT, int FMT>
static cudaError_t launch_dual_t(const void* x, int64_t rows, int64_t cols, int rule, int headroom,
                                 uint8_t* q_row, uint8_t* e8_row, uint8_t* q_colt, uint8_t* e8_colt,
                                 unsigned long long* cr, unsigned long long* cc, cudaStream_t s,
                                 int* launches) {
  auto kern = mx_dual_kernel<DT, FMT, DualCfg>;
  long long grid;
  cudaError_t e = tp_grid<DT, DualCfg>(reinterpret_cast<const void*>(kern), rows, cols, &grid);
  if (e != cudaSuccess) return e;
  CUtensorMap in, qm, qtm;
  e = tp_maps<DT>(x, rows, cols, q_row, q_colt, &in, &qm, &qtm);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)grid, kWThreads, DualCfg::kSmemBytes, s>>>(in, qm, qtm, rows, cols, rule, headroom, e8_row,
                                                              e8_colt, cr, cc);
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
  auto kern = cast_transpose_kernel<DT, FMT, CtCfg>;
  long long grid;
  cudaError_t e = tp_grid<DT, CtCfg>(reinterpret_cast<const void*>(kern), rows, cols, &grid);
  if (e != cudaSuccess) return e;
  CUtensorMap in, qm, qtm;
  e = tp_maps<DT>(x, rows, cols, q, qt, &in, &qm, &qtm);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)grid, kWThreads, CtCfg::kSmemBytes, s>>>(in, qm, qtm, rows, cols, st, mode, h);
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

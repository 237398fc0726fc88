// Per-warp TMA tile machinery shared by the column-wise MX cast and the
// fused transposes.
//
// Every warp runs its own pipeline: it streams 32-row x 128-byte sub-tiles
// (64 bf16 / 32 fp32 columns, 4 KiB) of a row-major [rows, cols] input
// through a few shared-memory stages filled by cp.async.bulk.tensor.2d with
// the 128-byte swizzle (chunk c of tile row r lands at chunk c ^ (r & 7)),
// one mbarrier per stage and bounded waits, and hands its 8-bit outputs to
// TMA tiled stores through swizzled staging buffers.  Warps never wait for
// one another.  With the swizzle, lane l can own tile row l (16-byte chunks)
// or the 32-bit word l of every row (a bf16 column pair or an fp32 column)
// without shared-memory bank conflicts.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "fp8q_device.cuh"
#include "fp8q_internal.cuh"
#include "mx_device.cuh"
#include "tma.cuh"

namespace fp8q {

constexpr int kWTileBytes = 32 * 128;                  // 32 rows x 128 bytes
constexpr int kWTileVec = kWTileBytes / 16;            // uint4 per sub-tile

// Pipeline shape of one kernel: S input stages per warp, OB output staging
// buffers of OUTB bytes per warp, CH row tiles per chunk, chunk order, at
// most MAXC resident CTAs per SM (0: as many as fit), whether the MX kernels
// count clipped elements (CNT false only for clip-free casts, which cannot
// clip) and whether they count every block (ALL) or only the blocks whose
// scaled maximum passes fmax, and W warps per CTA.  A CTA's warps start on W consecutive chunks
// and advance together by the grid's warp count, so with column strips
// first they always hold W adjacent column tiles of one row band: an SM
// whose warps all sit in one CTA reads and writes one wide band at a time.
template <int S, int OB, int CH, bool COLF, int OUTB, int MAXC = 0, bool CNT = true, int W = 4, bool ALL = false>
struct TpCfg {
  static_assert(S >= 2 && S <= 8, "input stages");
  static_assert(OB == 1 || OB == 2, "one or two output staging buffers");
  static_assert(CH >= 1 && CH <= 8, "the column E8M0 run is kept in one 64-bit word");
  static_assert(OUTB % 1024 == 0, "staging buffers keep the 1024-byte alignment of the swizzle");
  static_assert(W >= 1 && W <= 16, "warps per CTA");
  static constexpr int kStages = S, kOutBufs = OB, kChunk = CH, kOutBytes = OUTB;
  static constexpr bool kColFastest = COLF;      // chunk order: column tile fastest
  static constexpr int kMaxCtasPerSm = MAXC;
  static constexpr bool kClipCount = CNT;
  static constexpr bool kCountAll = CNT && ALL;
  static constexpr int kWarps = W, kThreads = 32 * W;
  // launch bounds: CTAs per SM the register budget must allow (at most 128
  // registers a thread, fewer CTAs for wider ones)
  static constexpr int kMinBlocks = W >= 16 ? 1 : 16 / W;
  static constexpr int kWarpBytes = S * kWTileBytes + OB * OUTB;
  static constexpr int kSmemBytes = W * kWarpBytes + 1024;   // + alignment slack
};

// True when no block of an MX cast can clip: under the round-up rule the
// scaled block maximum is at most fmax, and one or more binades of headroom
// keep it below fmax under every rule (the E clamp only lowers it further).
// Such casts run none of the per-element clip arithmetic, so their kernels
// take the pipeline shape of a lighter, more memory-bound pass.  The results
// do not depend on the shape.
inline bool mx_clip_free(int rule, int headroom) { return rule == FP8Q_MX_CEIL || headroom >= 1; }

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

// Max of |.| over 32 words as a depth-5 tree of one-instruction magnitude
// maxima (a serial chain would leave each thread waiting on 32 dependent
// operations).  Packed bf16 pairs (PAIRS, both lanes masked) or fp32 bit
// patterns.
template <bool PAIRS>
__device__ __forceinline__ uint32_t tree_absmax32(const uint32_t (&w)[32]) {
  constexpr int DT = PAIRS ? FP8Q_BF16 : FP8Q_F32;
  uint32_t t[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) t[i] = mag_max<DT>(w[2 * i], w[2 * i + 1]);
#pragma unroll
  for (int n = 8; n >= 1; n >>= 1)
#pragma unroll
    for (int i = 0; i < n; ++i) t[i] = mag_max<DT>(t[2 * i], t[2 * i + 1]);
  return t[0] & (PAIRS ? 0x7FFF7FFFu : 0x7FFFFFFFu);
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

// Byte b of row k of a staging tile with ROWB-byte rows in the swizzled
// layout of its tensor map (64-byte rows: 16-byte chunk c at c ^ ((k >> 1) & 3);
// 32-byte rows: c ^ ((k >> 2) & 1)).
template <int ROWB>
__device__ __forceinline__ int staged_byte(int k, int b) {
  const int sw = ROWB == 64 ? ((k >> 1) & 3) : ((k >> 2) & 1);
  return k * ROWB + ((((b >> 4) ^ sw)) << 4) + (b & 15);
}

// One MX column block (column HI of the lane's words): its 32 bytes into o,
// returns its E8M0 byte.  m = the block's max |x| bits.  With CNT the
// block's clipped elements are added to clip, tested per element when its
// scaled max passes fmax, or for every block with ALL (a block that cannot
// clip adds 0); a clip-free cast (no CNT) has nothing to count and carries
// no count code.
template <int FMT, int HI, bool CNT, bool ALL = false>
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
    if (CNT && (ALL || mx_block_may_clip<FMT>(m, E))) {
#pragma unroll
      for (int k = 0; k < 32; ++k) clip += clips<FMT>(__uint_as_float(half_bits<HI>(w[k])) * s) ? 1u : 0u;
    }
  }
  return ebyte;
}

// L2 policy for stores whose 32-byte sectors are completed over a long
// stretch of the kernel by many warps: evict-last keeps such partly
// written lines in L2 ahead of the streaming data.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// The E8M0 bytes of one column for the row tiles i0 .. i0 + n - 1 of a chunk
// (byte k of acc for row tile i0 + k), at e8 = the byte of row tile i0.  A
// full chunk at an address aligned to its size goes out as one store.  A
// column's 32-byte sector of E8M0 bytes (32 row tiles) is filled by 32 / CH
// chunks that different warps take at different times, so these stores
// carry the evict-last policy; with plain stores they cost the MX dual ~5 us
// (OCP rule, bf16 [16384, 8192], same box: 103.1 us plain, 98.3 us with the
// policy, 97 us with the stores left out).
template <int CH>
using E8Acc = typename std::conditional<(CH > 4), unsigned long long, uint32_t>::type;
template <int CH>
__device__ __forceinline__ void store_e8_run(uint8_t* e8, E8Acc<CH> acc, uint32_t n) {
  if (n == (uint32_t)CH && (CH == 4 || CH == 8) && (reinterpret_cast<uintptr_t>(e8) & (CH - 1)) == 0) {
    const uint64_t pol = l2_evict_last_policy();
    if (CH == 4)
      asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;" ::"l"(e8), "r"((uint32_t)acc), "l"(pol) : "memory");
    else
      asm volatile("st.global.L2::cache_hint.b64 [%0], %1, %2;" ::"l"(e8), "l"((unsigned long long)acc), "l"(pol)
                   : "memory");
    return;
  }
  for (uint32_t k = 0; k < n; ++k) e8[k] = (uint8_t)(acc >> (8 * k));
}

// Work order.  The sub-tiles form a grid of rtiles x ctiles (32 rows x
// tile_c columns each).  A chunk is CH consecutive row tiles of one
// column tile (fewer at the bottom edge); chunks are numbered row-chunk
// fastest (COLF false: the warps in flight together cover a band of
// adjacent column strips) or column-tile fastest (COLF true: a band of
// adjacent row chunks), and dealt to the warps round-robin (warp w takes
// chunks w, w + nwarps, ...).  Within a chunk a warp walks down the rows, so
// it can collect each column's CH transposed-scale bytes into one store.
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
  unsigned int* timeouts;        // counts barrier waits that ran out of time
  int tile_c;
  Cursor cur;                    // the sub-tile being processed
  Cursor next;                   // lane 0: the next sub-tile to issue

  __device__ __forceinline__ void setup(const CUtensorMap* m, uint4* st, uint64_t* f, uint32_t row_tiles,
                                        uint32_t col_tiles, int tc, unsigned int* timeout_counter) {
    map = m;
    timeouts = timeout_counter;
    stages = st;
    full = f;
    tile_c = tc;
    rtiles = row_tiles;
    const uint32_t rchunks = (row_tiles + kChunkR - 1) / kChunkR;
    nchunks = rchunks * col_tiles;
    nfast = kColF ? col_tiles : rchunks;
    stride = gridDim.x * C::kWarps;
    sq = stride / nfast;
    sr = stride % nfast;
    cur.v = blockIdx.x * C::kWarps + (threadIdx.x >> 5);
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
        atomicAdd(timeouts, 1u);
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
  __device__ __forceinline__ uint8_t* buf(uint32_t j) const { return base + (j % kOutBufs) * C::kOutBytes; }
  // Before writing buffer j: the store that last read it has read it.
  // Warp-collective.
  __device__ __forceinline__ void acquire() const {
    if ((threadIdx.x & 31) == 0) {
      bulk_wait_read<kOutBufs - 1>();
    }
    __syncwarp();
  }
  // Buffer j is written: copy it out, the row-major part (offset 0) through
  // qmap at (c0, r0) and, when qtmap is given, the transposed part (offset
  // 2048) through qtmap at (r0, c0).  Warp-collective.
  __device__ __forceinline__ void publish(uint32_t j, const CUtensorMap* qmap, const CUtensorMap* qtmap, int64_t r0,
                                         int64_t c0) const {
    fence_proxy_async();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
      tma_store_2d(qmap, buf(j), (int)c0, (int)r0);
      if (qtmap) tma_store_2d(qtmap, buf(j) + 2048, (int)r0, (int)c0);
      bulk_commit();
    }
  }
  // Before the warp leaves: its stores are complete.  Warp-collective.
  __device__ __forceinline__ void drain() const {
    if ((threadIdx.x & 31) == 0) bulk_wait_all();
    __syncwarp();
  }
};

}  // namespace fp8q

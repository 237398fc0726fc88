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
// Both run the per-warp pipeline of warp_tiles.cuh.  Lane l of a warp owns,
// per 32-row x 128-byte sub-tile:
//   A. row pass: row l, i.e. 2 (bf16) / 1 (fp32) 32-element row blocks, read
//      as 16-byte chunks, its 32 output bytes per block staged row-major;
//   B. column pass: bf16 columns 2l and 2l + 1 or fp32 column l, its 32
//      output bytes per column staged as one row of the transposed part.
//      The MX dual reads the column from the input tile (one 32-bit word per
//      row) and casts it with the column block's own scale; the per-tensor
//      cast reads back the bytes the row pass staged (same scale, same bytes).
// Both parts leave through TMA tiled stores.
#include <cuda.h>
#include <cuda_runtime.h>

#include "fp8q_device.cuh"
#include "fp8q_internal.cuh"
#include "state.cuh"
#include "tma.cuh"
#include "warp_tiles.cuh"

namespace fp8q {

// Pipeline shape of each kernel: TpCfg<input stages per warp, output
// staging buffers per warp, row tiles per chunk, column-strip-first chunk
// order, staging bytes, CTAs per SM (0: as many as fit), clip count, warps
// per CTA, count every block>.  The cast + transpose moves little arithmetic
// per byte: it runs one CTA of four warps per SM with six stages in flight
// per warp, which keeps the read stream and its two write streams closer to
// the DRAM rate than more, shallower warps do.  The MX dual runs twelve
// warps per SM (ten or fourteen measured slower), each with three input
// stages and one staging buffer, which is what shared memory allows, all in
// one CTA so that they work on twelve adjacent column tiles (a CTA's warps
// on distant chunks cost 5%).  It counts the clipped elements of every block
// without testing first whether the block can clip, under every rule: that
// straight-line form measured faster than the guarded count, than a
// clip-free kernel with no count, and than the guarded count on inputs where
// no block clips (round-up rule 100.4 -> 97.6 us, OCP on such inputs
// 103.8 -> 97.0 us, on tanh activations 97.8 -> 97.1 us; same box), and a
// block that cannot clip adds 0.  Each shape was chosen by same-box
// measurement on bf16 [16384, 8192].
using DualCfg = TpCfg<3, 1, 4, true, 4096, 1, true, 12, true>;
using CtCfg = TpCfg<6, 1, 4, true, 4096, 1>;
constexpr int kTpL2Promotion = 128;      // bytes the L2 fetches per input-tile request

static __device__ unsigned int g_tp_wait_timeouts;   // see fp8q_pipeline_status

cudaError_t read_tp_wait_timeouts(unsigned int* count) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(count, g_tp_wait_timeouts, sizeof(unsigned int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_tp_wait_timeouts, &zero, sizeof(unsigned int));
  return e;
}

// ---------------------------------------------------------------------------
// MX dual cast
// ---------------------------------------------------------------------------

template <int DT, int FMT, class C>
__global__ void __launch_bounds__(C::kThreads, C::kMinBlocks) mx_dual_kernel(
    const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap qmap,
    const __grid_constant__ CUtensorMap qtmap, int64_t rows, int64_t cols, int rule, int headroom,
    uint8_t* __restrict__ e8_row, uint8_t* __restrict__ e8_colt, unsigned long long* clipped_row,
    unsigned long long* clipped_col) {
  using G = TileGeom<DT>;
  constexpr int EPL = G::EPL, TILE_C = G::TILE_C, NG = G::NG;
  constexpr int QROWB = TILE_C;                      // bytes per row of the row-major part
  extern __shared__ __align__(1024) uint4 dyn_smem[];
  __shared__ __align__(8) uint64_t full[C::kWarps][C::kStages];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t ctiles = (uint32_t)((cols + TILE_C - 1) / TILE_C);
  uint8_t* region = warp_region<C>(dyn_smem, warp);
  WarpPipe<C> pipe;
  pipe.setup(&tmap, reinterpret_cast<uint4*>(region), full[warp], (uint32_t)(rows / 32), ctiles, TILE_C,
             &g_tp_wait_timeouts);
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
      uint32_t pm = mag_load<DT>(v[0]);
#pragma unroll
      for (int k = 1; k < NG; ++k) pm = mag_max<DT>(pm, mag_load<DT>(v[k]));
      const uint32_t m = mag_bits<DT>(pm);
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
        if (C::kClipCount && (C::kCountAll || mx_block_may_clip<FMT>(m, E))) {
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
        e8c0 |= (E8Acc<C::kChunk>)mx_column<FMT, 0, C::kClipCount, C::kCountAll>(w, pm << 16, rule, headroom, clip_c, o) << (8 * ci);
        stage32<32>(ob + 2048, 2 * lane, 0, o);
        e8c1 |= (E8Acc<C::kChunk>)mx_column<FMT, 1, C::kClipCount, C::kCountAll>(w, pm & 0xFFFF0000u, rule, headroom, clip_c, o) << (8 * ci);
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
        e8c0 |= (E8Acc<C::kChunk>)mx_column<FMT, 2, C::kClipCount, C::kCountAll>(w, tree_absmax32<false>(w), rule, headroom, clip_c, o) << (8 * ci);
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
__global__ void __launch_bounds__(C::kThreads, C::kMinBlocks) cast_transpose_kernel(
    const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap qmap,
    const __grid_constant__ CUtensorMap qtmap, int64_t rows, int64_t cols, DevState* st, int mode,
    GroupHeader h) {
  using G = TileGeom<DT>;
  constexpr int TILE_C = G::TILE_C, NG = G::NG;
  constexpr int QROWB = TILE_C;
  extern __shared__ __align__(1024) uint4 dyn_smem[];
  __shared__ __align__(8) uint64_t full[C::kWarps][C::kStages];
  __shared__ int s_e;
  __shared__ uint32_t s_nonfin[C::kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t ctiles = (uint32_t)((cols + TILE_C - 1) / TILE_C);
  const uint32_t ntiles = (uint32_t)(rows / 32) * ctiles;
  uint8_t* region = warp_region<C>(dyn_smem, warp);
  WarpPipe<C> pipe;
  pipe.setup(&tmap, reinterpret_cast<uint4*>(region), full[warp], (uint32_t)(rows / 32), ctiles, TILE_C,
             &g_tp_wait_timeouts);
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
      uint32_t pm = mag_load<DT>(v[0]);
#pragma unroll
      for (int k = 1; k < NG; ++k) pm = mag_max<DT>(pm, mag_load<DT>(v[k]));
      const uint32_t m = mag_bits<DT>(pm);
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
    lmax = max(lmax, tmax);
    pipe.release();                                  // the input stage is no longer read
    // B. transposed: q^T holds q's bytes, read back column-wise from the
    // row-major part and assembled with byte permutes
    __syncwarp();                                    // the row-major part is in place
    if (DT == FP8Q_BF16) {
      uint32_t a[8], bb[8];                          // columns 2l and 2l + 1, 4 rows per word
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        uint32_t u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) u[i] = *reinterpret_cast<const uint16_t*>(ob + staged_byte<64>(4 * m + i, 2 * lane));
        const uint32_t p01 = __byte_perm(u[0], u[1], 0x5410), p23 = __byte_perm(u[2], u[3], 0x5410);
        a[m] = __byte_perm(p01, p23, 0x6420);
        bb[m] = __byte_perm(p01, p23, 0x7531);
      }
      stage32<32>(ob + 2048, 2 * lane, 0, a);
      stage32<32>(ob + 2048, 2 * lane + 1, 0, bb);
    } else {
      uint32_t a[8];                                 // column l, 4 rows per word
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        uint32_t u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) u[i] = ob[staged_byte<32>(4 * m + i, lane)];
        a[m] = __byte_perm(__byte_perm(u[0], u[1], 0x0040), __byte_perm(u[2], u[3], 0x0040), 0x5410);
      }
      stage32<32>(ob + 2048, lane, 0, a);
    }
    out.publish(j, &qmap, &qtmap, r0, c0);
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
// Diagnostic of the per-warp pipeline's timeout path
// ---------------------------------------------------------------------------

// One warp sets up a pipeline over one sub-tile, initialises its barriers and
// issues no load, so its first wait cannot complete: the bounded wait gives
// up, counts the timeout and the warp stops (no tensor map is touched).
__global__ void warp_pipe_selftest_kernel() {
  using C = TpCfg<2, 1, 1, false, 2048>;
  __shared__ __align__(8) uint64_t full[C::kStages];
  WarpPipe<C> pipe;
  pipe.setup(nullptr, nullptr, full, 1u, 1u, 64, &g_tp_wait_timeouts);
  if ((threadIdx.x & 31) == 0) {
    for (int i = 0; i < C::kStages; ++i) mbar_init(&full[i], 1);
    fence_barrier_init();
  }
  __syncwarp();
  pipe.wait(0);
}

cudaError_t launch_warp_pipe_selftest(cudaStream_t s, int* launches) {
  warp_pipe_selftest_kernel<<<1, 32, 0, s>>>();
  ++*launches;
  return cudaGetLastError();
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
  cudaError_t e = kernel_occupancy(kern, C::kThreads, C::kSmemBytes, &occ);
  if (e != cudaSuccess) return e;
  if (C::kMaxCtasPerSm > 0 && occ > C::kMaxCtasPerSm) occ = C::kMaxCtasPerSm;
  long long gr = (long long)sm_count(device_of_current()) * occ;
  const long long need = (nchunks + C::kWarps - 1) / C::kWarps;
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
  cudaError_t e = encode_tile_map(in, x, DT == FP8Q_BF16, rows, cols, TILE_C, true, kTpL2Promotion);
  if (e == cudaSuccess) e = encode_byte_map(qmap, q, rows, cols, TILE_C, 32, TILE_C);
  if (e == cudaSuccess) e = encode_byte_map(qtmap, qt, cols, rows, 32, TILE_C, 32);
  return e;
}

template <int DT, int FMT, class C>
static cudaError_t launch_dual_c(const void* x, int64_t rows, int64_t cols, int rule, int headroom,
                                 uint8_t* q_row, uint8_t* e8_row, uint8_t* q_colt, uint8_t* e8_colt,
                                 unsigned long long* cr, unsigned long long* cc, cudaStream_t s,
                                 int* launches) {
  auto kern = mx_dual_kernel<DT, FMT, C>;
  long long grid;
  cudaError_t e = tp_grid<DT, C>(reinterpret_cast<const void*>(kern), rows, cols, &grid);
  if (e != cudaSuccess) return e;
  CUtensorMap in, qm, qtm;
  e = tp_maps<DT>(x, rows, cols, q_row, q_colt, &in, &qm, &qtm);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)grid, C::kThreads, C::kSmemBytes, s>>>(in, qm, qtm, rows, cols, rule, headroom, e8_row, e8_colt,
                                                        cr, cc);
  ++*launches;
  return cudaGetLastError();
}

template <int DT, int FMT>
static cudaError_t launch_dual_t(const void* x, int64_t rows, int64_t cols, int rule, int headroom,
                                 uint8_t* q_row, uint8_t* e8_row, uint8_t* q_colt, uint8_t* e8_colt,
                                 unsigned long long* cr, unsigned long long* cc, cudaStream_t s,
                                 int* launches) {
  return launch_dual_c<DT, FMT, DualCfg>(x, rows, cols, rule, headroom, q_row, e8_row, q_colt, e8_colt, cr, cc, s,
                                         launches);
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
  kern<<<(unsigned)grid, CtCfg::kThreads, CtCfg::kSmemBytes, s>>>(in, qm, qtm, rows, cols, st, mode, h);
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

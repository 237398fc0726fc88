// Fused per-tensor scaled cast over a group of tensors, one launch.
//
// Steps of one launch, per tensor ("Practice c06/E3" worked solution: the
// scale comes from the largest |x| over a window of steps; a power of two
// keeps that value at or below the format maximum with a margin):
//   1. every CTA that owns chunks of the tensor derives the exponent e from
//      the device-resident history window (or the current-scaling amax) --
//      integer compares only, no log2;
//   2. it streams its chunks: 128-bit loads of x, v = x * 2^e, saturating RNE
//      to FP8 two values per cvt, 128-bit (bf16) / 64-bit stores of q, and a
//      running max of |x| taken as an unsigned max of the abs bits;
//   3. warp + block reduction of (amax, clipped), one atomic each per CTA
//      and tensor segment;
//   4. the CTA whose atomic ticket completes the tensor pushes the amax into
//      the ring, publishes scale_inv / amax / clipped and resets the ticket.
// No CTA ever waits on another: there is no spin, flag or grid barrier.
//
// Work split: every tensor is cut into 32 KiB input chunks; the chunks of
// all tensors of the group form one index space cut into gridDim.x equal
// contiguous ranges, one per CTA.  A CTA therefore visits few tensors and
// flushes its partial results once per tensor.
//
// Launch: programmatic dependent launch.  Each CTA first waits until the
// preceding grid in the stream has completed and its writes are visible
// (griddepcontrol.wait), before any global access, then lets the next grid
// start launching (griddepcontrol.launch_dependents).  The next launch's
// set-up thus overlaps this grid's tail, and every dependency stays ordered
// (a cast reads the state the previous cast on the same handle left).  The
// grid is one wave (SMs x resident CTAs), so a dependent grid only takes SM
// slots that this one's finished CTAs free.
//
// This header holds the kernels and their launcher template; each group size
// (1, 32, 512 tensors per launch) is instantiated in its own translation
// unit (cast_g1.cu, cast_g32.cu, cast_g512.cu) so that they compile in
// parallel, and cast.cu dispatches to them.
#pragma once

#include <cuda_runtime.h>

#include "fp8q_device.cuh"
#include "fp8q_internal.cuh"
#include "state.cuh"

namespace fp8q {


__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <int DT>
struct Tr {
  static constexpr int EPL = DT == FP8Q_BF16 ? 8 : 4;   // elements per 16-B load
  static constexpr int ESZ = DT == FP8Q_BF16 ? 2 : 4;   // bytes per element
  static constexpr int CHUNK = kThreads * kUnroll * EPL;
};

// Load one chunk: slot u of thread tid holds elements
// [(u*kThreads + tid)*EPL, +EPL) of the chunk, so every warp-wide load
// covers 512 contiguous bytes.  Missing elements of a partial chunk are 0.
template <int DT, bool FULL>
__device__ __forceinline__ void load_chunk(const char* x, int64_t rem, uint4 (&r)[kUnroll]) {
  constexpr int EPL = Tr<DT>::EPL;
  const uint4* px = reinterpret_cast<const uint4*>(x) + threadIdx.x;
  if constexpr (FULL) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) r[u] = __ldcs(px + u * kThreads);
  } else {
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int64_t e0 = (int64_t)(u * kThreads + threadIdx.x) * EPL;
    if (e0 + EPL <= rem) {
      r[u] = __ldcs(px + u * kThreads);
    } else {
      uint32_t w[4] = {0u, 0u, 0u, 0u};
      for (int j = 0; j < EPL; ++j) {
        if (e0 + j < rem) {
          if (DT == FP8Q_BF16) {
            const uint32_t b = reinterpret_cast<const uint16_t*>(x)[e0 + j];
            w[j >> 1] |= b << ((j & 1) * 16);
          } else {
            w[j] = reinterpret_cast<const uint32_t*>(x)[e0 + j];
          }
        }
      }
      r[u] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  }
}

template <int DT>
__device__ __forceinline__ uint32_t chunk_absmax(const uint4 (&r)[kUnroll]) {
  uint32_t m = absmax_load<DT>(r[0]);
#pragma unroll
  for (int u = 1; u < kUnroll; ++u) m = absmax_merge<DT>(m, absmax_load<DT>(r[u]));
  return unpack_max<DT>(m);
}

// Cast a loaded chunk with scale s and store it.  m = the thread's abs-max
// over its slots (fp32 bits); the exact per-element pass runs only when m
// exceeds the no-clip bound (rare: clipping, Inf or NaN present).
template <int DT, int FMT, bool FULL, bool UF>
__device__ __forceinline__ void cast_store_chunk(const uint4 (&r)[kUnroll], uint8_t* q, int64_t rem,
                                                 float s, uint32_t m, uint32_t bound,
                                                 uint32_t ubound, uint32_t& clip,
                                                 uint32_t* s_nonfinite, uint32_t& under) {
  constexpr int EPL = Tr<DT>::EPL;
  const bool slow = m > bound;
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    uint2 o = cast_load<DT, FMT>(r[u], s);
    if (slow) fix_load<DT, FMT>(r[u], s, o, clip, s_nonfinite);
    if (UF) under += underflow_load<DT>(r[u], ubound);   // zero-filled tail slots count 0
    if (FULL) {
      if (DT == FP8Q_BF16) __stcs(reinterpret_cast<uint2*>(q) + threadIdx.x + u * kThreads, o);
      else __stcs(reinterpret_cast<unsigned int*>(q) + threadIdx.x + u * kThreads, o.x);
      continue;
    }
    const int64_t e0 = (int64_t)(u * kThreads + threadIdx.x) * EPL;
    if (e0 + EPL <= rem) {
      if (DT == FP8Q_BF16) __stcs(reinterpret_cast<uint2*>(q + e0), o);
      else __stcs(reinterpret_cast<unsigned int*>(q + e0), o.x);
    } else if (e0 < rem) {
      for (int j = 0; j < EPL && e0 + j < rem; ++j)
        q[e0 + j] = (uint8_t)(((j < 4 ? o.x : o.y) >> ((j & 3) * 8)) & 0xFFu);
    }
  }
}

__device__ __forceinline__ void block_reduce(uint32_t& mx, uint32_t& cnt, uint32_t* sm,
                                             uint32_t* sc) {
  mx = __reduce_max_sync(0xFFFFFFFFu, mx);
  cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) { sm[w] = mx; sc[w] = cnt; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < kThreads / 32; ++i) { mx = max(mx, sm[i]); cnt += sc[i]; }
  }
}

// Chunks [c0, c1) of tensor d (tensor-local chunk indices).
template <int DT, int FMT, bool UF>
__device__ void cast_segment(const TensorDesc& d, int c0, int c1, int mode, int* s_e,
                             uint32_t* red_m, uint32_t* red_c, uint32_t& lmax, uint32_t& lclip,
                             uint32_t* s_nonfin, uint32_t& lunder, int& e_out) {
  constexpr int CH = Tr<DT>::CHUNK, ESZ = Tr<DT>::ESZ;
  const char* x = reinterpret_cast<const char*>(d.x);
  if (mode == kCurrentLocal) {
    // the whole tensor is this one chunk: amax first, then the cast, from
    // the same registers
    uint4 r[kUnroll];
    load_chunk<DT, false>(x, d.n, r);
    const uint32_t m = chunk_absmax<DT>(r);
    uint32_t bm = m, dummy = 0;
    block_reduce(bm, dummy, red_m, red_c);
    if (threadIdx.x == 0) *s_e = state_exp(d.st, bm > 0x7F800000u ? 0x7FC00000u : bm);
    __syncthreads();
    const int e = *s_e;
    cast_store_chunk<DT, FMT, false, UF>(r, d.q, d.n, pow2f(e), m, no_clip_bound(FMT, e),
                                         UF ? underflow_bound(FMT, e) : 0u, lclip, s_nonfin, lunder);
    lmax = max(lmax, m);
    e_out = e;
    return;
  }
  if (threadIdx.x < 32) warp_exp(d.st, mode, s_e);
  __syncthreads();
  const int e = *s_e;
  const float s = pow2f(e);
  const uint32_t bound = no_clip_bound(FMT, e);
  const uint32_t ubound = UF ? underflow_bound(FMT, e) : 0u;
  for (int c = c0; c < c1; ++c) {
    const int64_t base = (int64_t)c * CH;
    const int64_t rem = d.n - base;
    uint4 r[kUnroll];
    if (rem >= CH) {
      load_chunk<DT, true>(x + base * ESZ, rem, r);
      const uint32_t m = chunk_absmax<DT>(r);
      lmax = max(lmax, m);
      cast_store_chunk<DT, FMT, true, UF>(r, d.q + base, rem, s, m, bound, ubound, lclip, s_nonfin, lunder);
    } else {
      load_chunk<DT, false>(x + base * ESZ, rem, r);
      const uint32_t m = chunk_absmax<DT>(r);
      lmax = max(lmax, m);
      cast_store_chunk<DT, FMT, false, UF>(r, d.q + base, rem, s, m, bound, ubound, lclip, s_nonfin, lunder);
    }
  }
  e_out = e;
}

template <int DT>
__device__ void amax_segment(const TensorDesc& d, int c0, int c1, uint32_t& lmax) {
  constexpr int CH = Tr<DT>::CHUNK, ESZ = Tr<DT>::ESZ;
  const char* x = reinterpret_cast<const char*>(d.x);
  for (int c = c0; c < c1; ++c) {
    const int64_t base = (int64_t)c * CH;
    const int64_t rem = d.n - base;
    uint4 r[kUnroll];
    if (rem >= CH) load_chunk<DT, true>(x + base * ESZ, rem, r);
    else load_chunk<DT, false>(x + base * ESZ, rem, r);
    lmax = max(lmax, chunk_absmax<DT>(r));
  }
}

// Contiguous chunk range of this CTA and the tensor holding its first chunk.
template <int MAXT>
__device__ __forceinline__ int first_tensor(const GroupParams<MAXT>& p, int c) {
  int lo = 0, hi = p.h.count - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.d[mid].chunk_begin <= c) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <int MAXT, bool UF>
__global__ void __launch_bounds__(kThreads, UF ? 3 : 4) cast_group_kernel(const __grid_constant__ GroupParams<MAXT> p) {
  __shared__ int s_e;
  __shared__ uint32_t s_nonfin;                   // non-finite inputs of the current segment
  __shared__ uint32_t red_m[kThreads / 32], red_c[kThreads / 32], red_u[kThreads / 32];
  if (threadIdx.x == 0) s_nonfin = 0u;            // published by the first __syncthreads below
  pdl_wait();
  pdl_launch_dependents();
  const int total = p.h.total_chunks;
  int c = (int)(((long long)blockIdx.x * total) / gridDim.x);
  const int c_end = (int)(((long long)(blockIdx.x + 1) * total) / gridDim.x);
  if (c >= c_end) return;
  int t = first_tensor(p, c);
  while (c < c_end) {
    const TensorDesc& d = p.d[t];
    const int t_begin = d.chunk_begin;
    const int t_end = (t + 1 < p.h.count) ? p.d[t + 1].chunk_begin : total;
    const int seg_end = min(c_end, t_end);
    const int mode = (d.flags >> 2) & 3;
    uint32_t lmax = 0, lclip = 0, lunder = 0;
    int e = 0;
    const int c0 = c - t_begin, c1 = seg_end - t_begin;
    switch (d.flags & 3) {
      case 0: cast_segment<FP8Q_F32, FP8Q_E4M3, UF>(d, c0, c1, mode, &s_e, red_m, red_c, lmax, lclip, &s_nonfin, lunder, e); break;
      case 1: cast_segment<FP8Q_BF16, FP8Q_E4M3, UF>(d, c0, c1, mode, &s_e, red_m, red_c, lmax, lclip, &s_nonfin, lunder, e); break;
      case 2: cast_segment<FP8Q_F32, FP8Q_E5M2, UF>(d, c0, c1, mode, &s_e, red_m, red_c, lmax, lclip, &s_nonfin, lunder, e); break;
      default: cast_segment<FP8Q_BF16, FP8Q_E5M2, UF>(d, c0, c1, mode, &s_e, red_m, red_c, lmax, lclip, &s_nonfin, lunder, e); break;
    }
    __syncthreads();                       // red_* reuse after the local-mode reduction
    block_reduce(lmax, lclip, red_m, red_c);
    if (UF) {
      lunder = __reduce_add_sync(0xFFFFFFFFu, lunder);
      if ((threadIdx.x & 31) == 0) red_u[threadIdx.x >> 5] = lunder;
      __syncthreads();
      if (threadIdx.x == 0)
        for (int i = 1; i < kThreads / 32; ++i) lunder += red_u[i];
    }
    if (threadIdx.x == 0) {
      DevState* st = d.st;
      const uint32_t lnonfin = s_nonfin;   // all slow-path adds happened before the reduction's barrier
      s_nonfin = 0u;
      if (c == t_begin && seg_end == t_end) {
        // this CTA holds the whole tensor: its totals are final, no
        // accumulator or ticket round trip
        publish_and_advance(st, p.h, t, e, lmax, lclip, lnonfin, UF ? lunder : 0u);
      } else {
        if (lmax) atomicMax(&st->amax_acc, lmax);
        if (lclip) atomicAdd(&st->clip_acc, (unsigned long long)lclip);
        if (lnonfin) atomicAdd(&st->nonfinite_acc, (unsigned long long)lnonfin);
        if (UF && lunder) atomicAdd(&st->underflow_acc, (unsigned long long)lunder);
        __threadfence();
        const unsigned done = (unsigned)(seg_end - c);
        const unsigned prev = atomicAdd(&st->ticket, done);
        if (prev + done == (unsigned)(t_end - t_begin)) finish_tensor(st, p.h, t, e);
      }
    }
    __syncthreads();
    c = seg_end;
    ++t;
  }
}

template <int MAXT>
__global__ void __launch_bounds__(kThreads, 4) amax_group_kernel(const __grid_constant__ GroupParams<MAXT> p) {
  __shared__ uint32_t red_m[kThreads / 32], red_c[kThreads / 32];
  pdl_wait();
  pdl_launch_dependents();
  const int total = p.h.total_chunks;
  int c = (int)(((long long)blockIdx.x * total) / gridDim.x);
  const int c_end = (int)(((long long)(blockIdx.x + 1) * total) / gridDim.x);
  if (c >= c_end) return;
  int t = first_tensor(p, c);
  while (c < c_end) {
    const TensorDesc& d = p.d[t];
    const int t_begin = d.chunk_begin;
    const int t_end = (t + 1 < p.h.count) ? p.d[t + 1].chunk_begin : total;
    const int seg_end = min(c_end, t_end);
    uint32_t lmax = 0, dummy = 0;
    if (d.flags & 1) amax_segment<FP8Q_BF16>(d, c - t_begin, seg_end - t_begin, lmax);
    else amax_segment<FP8Q_F32>(d, c - t_begin, seg_end - t_begin, lmax);
    block_reduce(lmax, dummy, red_m, red_c);
    if (threadIdx.x == 0 && lmax) atomicMax(&d.st->pre_amax, lmax);
    __syncthreads();
    c = seg_end;
    ++t;
  }
}

// ---- host-side launch ------------------------------------------------------

template <int MAXT, int KIND>   // KIND 0: amax pre-pass, 1: cast, 2: cast + underflow count
cudaError_t launch_group_t(const GroupHeader& h, const TensorDesc* d, int count,
                                  cudaStream_t s, int* launches) {
  GroupParams<MAXT> p;
  p.h = h;
  p.h.count = count;
  for (int i = 0; i < count; ++i) p.d[i] = d[i];
  auto kern = KIND == 0 ? amax_group_kernel<MAXT>
                        : (KIND == 1 ? cast_group_kernel<MAXT, false> : cast_group_kernel<MAXT, true>);
  int occ = 1;
  cudaError_t oe = kernel_occupancy(reinterpret_cast<const void*>(kern), kThreads, 0, &occ);
  if (oe != cudaSuccess) return oe;
  const int dev = device_of_current();
  long long grid = (long long)sm_count(dev) * occ;
  if (grid > h.total_chunks) grid = h.total_chunks;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  ++*launches;
  return e != cudaSuccess ? e : cudaGetLastError();
}

// The instantiations, one translation unit per group size.
#define FP8Q_CAST_GROUP_INSTANCES(SPEC, MAXT)                                                          \
  SPEC template cudaError_t launch_group_t<MAXT, 0>(const GroupHeader&, const TensorDesc*, int, cudaStream_t, int*); \
  SPEC template cudaError_t launch_group_t<MAXT, 1>(const GroupHeader&, const TensorDesc*, int, cudaStream_t, int*); \
  SPEC template cudaError_t launch_group_t<MAXT, 2>(const GroupHeader&, const TensorDesc*, int, cudaStream_t, int*);

}  // namespace fp8q

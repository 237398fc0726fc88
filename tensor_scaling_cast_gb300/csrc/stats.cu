// Dequantised-error statistics of a cast, off the timed path ("what actually
// breaks low precision training", "What the measurements said": how much the
// cast changes a tensor and which way it points, measured separately).
//
// deq = decode(q) * scale, scale = scale_inv (per tensor) or 2^E (MX block);
// over the elements with a finite input (and, for MX, a non-NaN block):
//   out[0] = mean((deq - x)^2), out[1] = mean(deq - x), out[2] = count.
// Differences and squares are formed in fp64.  Each CTA writes its partial
// sums to a scratch row; a one-CTA kernel adds the rows in index order, so the
// result does not depend on scheduling.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "fp8q_device.cuh"
#include "fp8q_internal.cuh"

namespace fp8q {

constexpr int kStatThreads = 256;

// Value of an FP8 code (finite codes only are ever read here).
template <int FMT>
__device__ float decode_code(uint32_t c) {
  constexpr int MB = FMT == FP8Q_E4M3 ? 3 : 2;
  constexpr int BIAS = FMT == FP8Q_E4M3 ? 7 : 15;
  const uint32_t ef = (c >> MB) & (FMT == FP8Q_E4M3 ? 0xFu : 0x1Fu);
  const uint32_t mf = c & ((1u << MB) - 1u);
  float v = ef ? ldexpf((float)((1u << MB) | mf), (int)ef - BIAS - MB)
               : ldexpf((float)mf, 1 - BIAS - MB);
  return (c & 0x80u) ? -v : v;
}

template <int DT, int FMT, bool MX>
__global__ void __launch_bounds__(kStatThreads) stats_partial_kernel(
    const char* __restrict__ x, int64_t n, const uint8_t* __restrict__ q,
    const float* __restrict__ scale_inv, const uint8_t* __restrict__ e8m0,
    double* __restrict__ partial) {
  __shared__ float lut[256];
  __shared__ double s1[kStatThreads / 32], s2[kStatThreads / 32];
  __shared__ unsigned long long sc[kStatThreads / 32];
  for (int c = threadIdx.x; c < 256; c += kStatThreads) lut[c] = decode_code<FMT>((uint32_t)c);
  __syncthreads();
  const double sinv = MX ? 1.0 : (double)__ldg(scale_inv);
  double a1 = 0.0, a2 = 0.0;
  unsigned long long cnt = 0;
  for (int64_t i = (int64_t)blockIdx.x * kStatThreads + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * kStatThreads) {
    const uint32_t b = DT == FP8Q_BF16 ? ((uint32_t)reinterpret_cast<const uint16_t*>(x)[i]) << 16
                                       : reinterpret_cast<const uint32_t*>(x)[i];
    if ((b & 0x7FFFFFFFu) >= 0x7F800000u) continue;
    double sc_i = sinv;
    if (MX) {
      const uint32_t eb = e8m0[i >> 5];
      if (eb == 0xFFu) continue;
      sc_i = ldexp(1.0, (int)eb - 127);
    }
    const double d = (double)lut[q[i]] * sc_i - (double)__uint_as_float(b);
    a1 += d;
    a2 += d * d;
    ++cnt;
  }
  for (int o = 16; o > 0; o >>= 1) {
    a1 += __shfl_xor_sync(0xFFFFFFFFu, a1, o);
    a2 += __shfl_xor_sync(0xFFFFFFFFu, a2, o);
    cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, o);
  }
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) { s1[w] = a1; s2[w] = a2; sc[w] = cnt; }
  __syncthreads();
  if (threadIdx.x == 0) {
    double t1 = 0.0, t2 = 0.0;
    unsigned long long tc = 0;
    for (int i = 0; i < kStatThreads / 32; ++i) { t1 += s1[i]; t2 += s2[i]; tc += sc[i]; }
    partial[3 * blockIdx.x + 0] = t2;
    partial[3 * blockIdx.x + 1] = t1;
    partial[3 * blockIdx.x + 2] = (double)tc;
  }
}

__global__ void stats_final_kernel(const double* __restrict__ partial, int rows, double* out) {
  if (threadIdx.x != 0) return;
  double t2 = 0.0, t1 = 0.0, tc = 0.0;
  for (int i = 0; i < rows; ++i) {
    t2 += partial[3 * i];
    t1 += partial[3 * i + 1];
    tc += partial[3 * i + 2];
  }
  out[0] = tc > 0.0 ? t2 / tc : 0.0;
  out[1] = tc > 0.0 ? t1 / tc : 0.0;
  out[2] = tc;
}

template <int DT, int FMT, bool MX>
static void launch_partial(const void* x, int64_t n, const uint8_t* q, const float* scale_inv,
                           const uint8_t* e8m0, double* partial, int grid, cudaStream_t s) {
  stats_partial_kernel<DT, FMT, MX><<<grid, kStatThreads, 0, s>>>(
      reinterpret_cast<const char*>(x), n, q, scale_inv, e8m0, partial);
}

cudaError_t launch_stats(const void* x, int dtype, int64_t n, const uint8_t* q, int format,
                         const float* scale_inv, const uint8_t* e8m0, double* out, cudaStream_t s,
                         int* launches) {
  if (n == 0) return cudaMemsetAsync(out, 0, 3 * sizeof(double), s);   // 0.0 is all-zero bits
  // fixed grid per device: the reduction order, hence the result, is
  // reproducible on a given GPU
  const int grid = sm_count(device_of_current()) * 4;
  double* partial = nullptr;
  cudaError_t err = cudaMallocAsync(reinterpret_cast<void**>(&partial),
                                    sizeof(double) * 3 * (size_t)grid, s);
  if (err != cudaSuccess) return err;
  const bool mx = e8m0 != nullptr;
  const int key = (dtype == FP8Q_BF16 ? 1 : 0) | (format == FP8Q_E5M2 ? 2 : 0) | (mx ? 4 : 0);
  switch (key) {
    case 0: launch_partial<FP8Q_F32, FP8Q_E4M3, false>(x, n, q, scale_inv, e8m0, partial, grid, s); break;
    case 1: launch_partial<FP8Q_BF16, FP8Q_E4M3, false>(x, n, q, scale_inv, e8m0, partial, grid, s); break;
    case 2: launch_partial<FP8Q_F32, FP8Q_E5M2, false>(x, n, q, scale_inv, e8m0, partial, grid, s); break;
    case 3: launch_partial<FP8Q_BF16, FP8Q_E5M2, false>(x, n, q, scale_inv, e8m0, partial, grid, s); break;
    case 4: launch_partial<FP8Q_F32, FP8Q_E4M3, true>(x, n, q, scale_inv, e8m0, partial, grid, s); break;
    case 5: launch_partial<FP8Q_BF16, FP8Q_E4M3, true>(x, n, q, scale_inv, e8m0, partial, grid, s); break;
    case 6: launch_partial<FP8Q_F32, FP8Q_E5M2, true>(x, n, q, scale_inv, e8m0, partial, grid, s); break;
    default: launch_partial<FP8Q_BF16, FP8Q_E5M2, true>(x, n, q, scale_inv, e8m0, partial, grid, s); break;
  }
  ++*launches;
  err = cudaGetLastError();
  if (err == cudaSuccess) {
    stats_final_kernel<<<1, 32, 0, s>>>(partial, grid, out);
    ++*launches;
    err = cudaGetLastError();
  }
  const cudaError_t ferr = cudaFreeAsync(partial, s);
  return err != cudaSuccess ? err : ferr;
}

}  // namespace fp8q

// ---- allocation-free variant of the per-tensor statistics ------------------
//
// For callers that cannot allocate device memory when they want the
// statistics (their own allocator owns the device's memory, they run after
// an out-of-memory error, or an allocation would stall a latency-bound
// loop).  The per-CTA partial sums go to this fixed array instead of a
// cudaMallocAsync block, one row of three doubles per CTA.  The grid is the
// allocating variant's (4 CTAs per SM), raised to one CTA per 2^20 elements
// for larger tensors, and never above the array's 4096 rows: each CTA
// grid-strides over the tensor, so n <= 4096 * 2^20 keeps a CTA's share at
// most 2^20 elements.  Every row the final kernel reads (rows 0 .. grid-1)
// is written earlier in the same call, so nothing needs clearing between
// calls.
namespace fp8q {

constexpr int kNoAllocRows = FP8Q_STATS_NOALLOC_ROWS;
constexpr int64_t kNoAllocSlab = int64_t(1) << 20;
static_assert(FP8Q_STATS_NOALLOC_MAX_N == kNoAllocRows * kNoAllocSlab, "limit and rows disagree");

static __device__ __align__(256) double g_stats_scratch[3 * kNoAllocRows];

// Device address of g_stats_scratch for each device (the host-side name is
// only a stand-in), looked up with that device current on the first call,
// and again when the device's context is no longer the one the address was
// taken in (a caller's cudaDeviceReset re-creates the context and reloads
// the module, which moves the array).  Contexts are told apart by the
// driver's per-process unique context id.
struct ScratchEntry {
  unsigned long long ctx_id;
  double* ptr;
};
static std::mutex g_scratch_mu;
static ScratchEntry g_scratch[128] = {};

unsigned long long current_context_id();   // api.cu

static cudaError_t stats_scratch(int device, double** out) {
  if (device < 0 || device >= 128) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  ScratchEntry& en = g_scratch[device];
  const unsigned long long id = current_context_id();
  if (en.ptr == nullptr || id == 0 || id != en.ctx_id) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_stats_scratch);   // makes the context current
    if (e != cudaSuccess) return e;
    en.ptr = static_cast<double*>(p);
    en.ctx_id = current_context_id();
  }
  *out = en.ptr;
  return cudaSuccess;
}

}  // namespace fp8q

extern "C" FP8Q_API int fp8q_error_stats_noalloc(const void* x, int dtype, int64_t n,
                                                 const uint8_t* q, int format,
                                                 const float* d_scale_inv, double* d_out,
                                                 void* stream) {
  FP8Q_TRACE_CALL();
  using namespace fp8q;
  if (dtype != FP8Q_F32 && dtype != FP8Q_BF16) return FP8Q_EDTYPE;
  if (format != FP8Q_E4M3 && format != FP8Q_E5M2) return FP8Q_EDTYPE;
  if (n < 0 || !d_out || !d_scale_inv || (n > 0 && (!x || !q))) return FP8Q_EINVAL;
  if (n > FP8Q_STATS_NOALLOC_MAX_N) return FP8Q_ESIZE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (n == 0) {
    const cudaError_t e = cudaMemsetAsync(d_out, 0, 3 * sizeof(double), s);
    return e == cudaSuccess ? FP8Q_OK : record_cuda_error(e);
  }
  double* partial = nullptr;
  cudaError_t e = stats_scratch(device_of_current(), &partial);
  if (e != cudaSuccess) return record_cuda_error(e);
  const int64_t slabs = (n + kNoAllocSlab - 1) / kNoAllocSlab;
  const int grid = (int)std::min<int64_t>(
      kNoAllocRows, std::max<int64_t>(slabs, (int64_t)sm_count(device_of_current()) * 4));
  const int key = (dtype == FP8Q_BF16 ? 1 : 0) | (format == FP8Q_E5M2 ? 2 : 0);
  switch (key) {
    case 0: launch_partial<FP8Q_F32, FP8Q_E4M3, false>(x, n, q, d_scale_inv, nullptr, partial, grid, s); break;
    case 1: launch_partial<FP8Q_BF16, FP8Q_E4M3, false>(x, n, q, d_scale_inv, nullptr, partial, grid, s); break;
    case 2: launch_partial<FP8Q_F32, FP8Q_E5M2, false>(x, n, q, d_scale_inv, nullptr, partial, grid, s); break;
    default: launch_partial<FP8Q_BF16, FP8Q_E5M2, false>(x, n, q, d_scale_inv, nullptr, partial, grid, s); break;
  }
  e = cudaGetLastError();
  if (e == cudaSuccess) {
    stats_final_kernel<<<1, 32, 0, s>>>(partial, grid, d_out);
    e = cudaGetLastError();
  }
  note_launches(2);
  return e == cudaSuccess ? FP8Q_OK : record_cuda_error(e);
}


// C ABI of libfp8q: argument checks, handle lifecycle, launch planning.
// Every entry point returns a status; nothing throws across the ABI.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "fp8q.h"
#include "fp8q_internal.cuh"
#include "mx_device.cuh"

namespace fp8q {

static std::atomic<long long> g_launches{0};
static thread_local char g_cuda_err[256] = "";

static int fail_cuda(cudaError_t e) {
  std::snprintf(g_cuda_err, sizeof g_cuda_err, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return FP8Q_ECUDA;
}

int record_cuda_error(cudaError_t e) { return fail_cuda(e); }

void note_launches(int k) { g_launches += k; }

int device_of_current() {
  int d = 0;
  cudaGetDevice(&d);
  return d;
}

// Id of the calling thread's current CUDA context (0 if none or unknown):
// what a device-resident address or a per-function attribute is valid for.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext c = nullptr;
  if (get_current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
  unsigned long long id = 0;
  return get_id(c, &id) == CUDA_SUCCESS ? id : 0;
}

// Resident CTAs per SM of a kernel at `threads` threads and `smem` bytes of
// dynamic shared memory, computed once per (kernel, size, device, context);
// the kernel's dynamic shared-memory limit is raised to `smem` first when
// that exceeds the 48 KiB default (an attribute of the context, so a
// re-created context sets it again).  Thread-safe.
cudaError_t kernel_occupancy(const void* kernel, int threads, int smem, int* occ) {
  struct Entry { const void* k; int threads, smem, device; unsigned long long ctx; int occ; };
  static std::mutex mu;
  static std::vector<Entry> cache;
  const int device = device_of_current();
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lk(mu);
  for (const Entry& en : cache)
    if (en.k == kernel && en.threads == threads && en.smem == smem && en.device == device && ctx != 0 &&
        en.ctx == ctx) {
      *occ = en.occ;
      return cudaSuccess;
    }
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  int v = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kernel, threads, (size_t)smem) != cudaSuccess || v < 1)
    v = 1;
  cache.push_back({kernel, threads, smem, device, ctx, v});
  *occ = v;
  return cudaSuccess;
}

int sm_count(int device) {
  static std::mutex mu;
  static int cache[128] = {0};
  if (device < 0 || device >= 128) return 1;
  std::lock_guard<std::mutex> lk(mu);
  if (cache[device] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || v < 1) v = 1;
    cache[device] = v;
  }
  return cache[device];
}

}  // namespace fp8q

using namespace fp8q;

static const uint32_t kMagic = 0xF8A5C0DEu;

struct fp8q_state {
  uint32_t magic;
  int format, window, margin, hyst;
  int estimator, interval;
  float alpha;
  long long host_casts;     // casts enqueued, mirrored on the host
  int device;
  DevState* dev;
  int host_count;           // valid history entries, mirrored on the host
  cudaEvent_t last;         // recorded after each cast on its stream
  bool has_last;
};

static bool handle_ok(fp8q_handle h) { return h != nullptr && h->magic == kMagic; }
static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool dtype_ok(int d) { return d == FP8Q_F32 || d == FP8Q_BF16; }
static bool format_ok(int f) { return f == FP8Q_E4M3 || f == FP8Q_E5M2; }

static int check_device(fp8q_handle h) {
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return fail_cuda(e);
  return d == h->device ? FP8Q_OK : FP8Q_EDEVICE;
}

// Wait for the handle's last cast (before a host read or write of its state).
static int wait_last(fp8q_handle h) {
  if (!h->has_last) return FP8Q_OK;
  cudaError_t e = cudaEventSynchronize(h->last);
  return e == cudaSuccess ? FP8Q_OK : fail_cuda(e);
}

// Is s capturing into a CUDA graph?
static bool stream_capturing(cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return cs == cudaStreamCaptureStatusActive;
}

// Would the handle's next cast be its first one under an estimator that
// takes current scaling only then (window > 0, or the smoothed average)?
// Such a cast picks its path on the host from that fact, so it must not be
// captured into a graph whose replays come later.
static bool first_windowed_cast(fp8q_handle h) {
  return h->estimator == FP8Q_EST_SMOOTHED ? h->host_casts == 0 : (h->window > 0 && h->host_count == 0);
}

// After a cast enqueued on s: remember it for the host reads of the state.
// A cast captured into a graph is not recorded (its replays are the
// caller's to wait for).
static int record_last(fp8q_handle h, cudaStream_t s) {
  if (stream_capturing(s)) return FP8Q_OK;
  cudaError_t e = cudaEventRecord(h->last, s);
  if (e != cudaSuccess) return fail_cuda(e);
  h->has_last = true;
  return FP8Q_OK;
}

extern "C" {

FP8Q_API const char* fp8q_strerror(int code) {
  switch (code) {
    case FP8Q_OK: return "ok";
    case FP8Q_EINVAL: return "invalid argument";
    case FP8Q_EALIGN: return "pointer not 16-byte aligned";
    case FP8Q_EDTYPE: return "unsupported dtype or format";
    case FP8Q_ECUDA: return "CUDA error";
    case FP8Q_EHANDLE: return "invalid handle";
    case FP8Q_ENOMEM: return "out of memory";
    case FP8Q_EDEVICE: return "handle used on another device";
    case FP8Q_ESIZE: return "size above the fixed scratch limit";
    default: return "unknown status";
  }
}

FP8Q_API const char* fp8q_last_cuda_error(void) { return g_cuda_err; }

FP8Q_API int fp8q_pipeline_selftest(void* stream) {
  FP8Q_TRACE_CALL();
  int launches = 0;
  cudaError_t e = launch_pipeline_selftest(reinterpret_cast<cudaStream_t>(stream), &launches);
  if (e == cudaSuccess) e = launch_warp_pipe_selftest(reinterpret_cast<cudaStream_t>(stream), &launches);
  g_launches += launches;
  return e == cudaSuccess ? FP8Q_OK : fail_cuda(e);
}

FP8Q_API int fp8q_pipeline_status(unsigned int* timed_out_waits) {
  FP8Q_TRACE_CALL();
  if (!timed_out_waits) return FP8Q_EINVAL;
  unsigned int a = 0, b = 0;
  cudaError_t e = read_wait_timeouts(&a);
  if (e == cudaSuccess) e = read_tp_wait_timeouts(&b);
  *timed_out_waits = a + b;
  return e == cudaSuccess ? FP8Q_OK : fail_cuda(e);
}

FP8Q_API long long fp8q_launch_count(void) { return g_launches.load(); }

FP8Q_API int fp8q_create_ex(int format, int window, int margin_bits, int hysteresis_bits,
                            int estimator, float alpha, int interval, fp8q_handle* out) {
  FP8Q_TRACE_CALL();
  if (!out) return FP8Q_EINVAL;
  *out = nullptr;
  if (!format_ok(format)) return FP8Q_EDTYPE;
  if (window < 0 || window > FP8Q_MAX_WINDOW || margin_bits < 0 || margin_bits > 16 ||
      hysteresis_bits < 0 || hysteresis_bits > 16)
    return FP8Q_EINVAL;
  if (estimator != FP8Q_EST_MAX_WINDOW && estimator != FP8Q_EST_SMOOTHED) return FP8Q_EINVAL;
  if (!(alpha > 0.0f && alpha <= 1.0f) || interval < 1) return FP8Q_EINVAL;
  fp8q_state* h = new (std::nothrow) fp8q_state();
  if (!h) return FP8Q_ENOMEM;
  h->format = format;
  h->window = window;
  h->margin = margin_bits;
  h->hyst = hysteresis_bits;
  h->estimator = estimator;
  h->alpha = alpha;
  h->interval = interval;
  h->host_count = 0;
  h->host_casts = 0;
  h->has_last = false;
  cudaError_t e = cudaGetDevice(&h->device);
  if (e != cudaSuccess) { delete h; return fail_cuda(e); }
  e = cudaMalloc(reinterpret_cast<void**>(&h->dev), sizeof(DevState));
  if (e != cudaSuccess) { delete h; return e == cudaErrorMemoryAllocation ? FP8Q_ENOMEM : fail_cuda(e); }
  DevState init;
  std::memset(&init, 0, sizeof init);
  init.format = format;
  init.window = window;
  init.margin = margin_bits;
  init.hyst = hysteresis_bits;
  init.estimator = estimator;
  init.alpha = alpha;
  init.interval = interval;
  e = cudaMemcpy(h->dev, &init, sizeof init, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->last, cudaEventDisableTiming);
  if (e != cudaSuccess) { cudaFree(h->dev); delete h; return fail_cuda(e); }
  h->magic = kMagic;
  *out = h;
  return FP8Q_OK;
}

FP8Q_API int fp8q_create(int format, int window, int margin_bits, int hysteresis_bits,
                         fp8q_handle* out) {
  FP8Q_TRACE_CALL();
  return fp8q_create_ex(format, window, margin_bits, hysteresis_bits, FP8Q_EST_MAX_WINDOW, 1.0f,
                        1, out);
}

FP8Q_API int fp8q_destroy(fp8q_handle h) {
  FP8Q_TRACE_CALL();
  if (h == nullptr) return FP8Q_OK;
  if (!handle_ok(h)) return FP8Q_EHANDLE;
  int dev = 0;
  cudaGetDevice(&dev);
  cudaSetDevice(h->device);
  if (h->has_last) cudaEventSynchronize(h->last);
  cudaEventDestroy(h->last);
  cudaError_t e = cudaFree(h->dev);
  cudaSetDevice(dev);
  h->magic = 0;
  delete h;
  return e == cudaSuccess ? FP8Q_OK : fail_cuda(e);
}

// Build the descriptors of a group, launch the current-scaling pre-pass for
// the tensors that need it, then the fused cast.
static int plan_and_launch(const fp8q_handle* hs, const void* const* xs, const int* dtypes,
                           const int64_t* ns, uint8_t* const* qs, float* d_scale_inv,
                           float* d_amax, unsigned long long* d_clipped,
                           unsigned long long* d_nonfinite, unsigned long long* d_underflow,
                           int count, cudaStream_t s) {
  if (stream_capturing(s))
    for (int i = 0; i < count; ++i)
      if (first_windowed_cast(hs[i])) return FP8Q_EINVAL;
  for (int base = 0; base < count; base += kMaxGroup) {
    const int m = std::min(kMaxGroup, count - base);
    std::vector<TensorDesc> all(m), pre;
    long long chunks = 0, pre_chunks = 0;
    for (int i = 0; i < m; ++i) {
      const fp8q_handle h = hs[base + i];
      const int dt = dtypes[base + i];
      const int64_t n = ns[base + i];
      const int64_t ce = chunk_elems(dt);
      const long long nch = std::max<long long>(1, (n + ce - 1) / ce);
      int mode = kDelayed;
      const bool current = h->estimator == FP8Q_EST_SMOOTHED ? h->host_casts == 0
                                                             : (h->window == 0 || h->host_count == 0);
      if (current) mode = (n <= ce) ? kCurrentLocal : kCurrentPre;
      TensorDesc d;
      d.x = xs[base + i];
      d.q = qs[base + i];
      d.n = n;
      d.st = h->dev;
      d.chunk_begin = (int32_t)chunks;
      d.flags = (dt == FP8Q_BF16 ? 1 : 0) | (h->format == FP8Q_E5M2 ? 2 : 0) | (mode << 2);
      all[i] = d;
      chunks += nch;
      if (mode == kCurrentPre) {
        TensorDesc p = d;
        p.chunk_begin = (int32_t)pre_chunks;
        pre.push_back(p);
        pre_chunks += nch;
      }
    }
    if (chunks > 0x7FFFFFFFll) return FP8Q_EINVAL;
    int launches = 0;
    GroupHeader gh;
    std::memset(&gh, 0, sizeof gh);
    if (!pre.empty()) {
      gh.total_chunks = (int32_t)pre_chunks;
      cudaError_t e = launch_amax_group(gh, pre.data(), (int)pre.size(), s, &launches);
      g_launches += launches;
      if (e != cudaSuccess) return fail_cuda(e);
      launches = 0;
    }
    gh.scale_inv = d_scale_inv;
    gh.amax = d_amax;
    gh.clipped = d_clipped;
    gh.nonfinite = d_nonfinite;
    gh.underflow = d_underflow;
    gh.total_chunks = (int32_t)chunks;
    gh.out_offset = base;
    cudaError_t e = launch_cast_group(gh, all.data(), m, s, &launches);
    g_launches += launches;
    if (e != cudaSuccess) return fail_cuda(e);
    for (int i = 0; i < m; ++i) {
      fp8q_handle h = hs[base + i];
      if (h->window > 0 && h->host_count < h->window) h->host_count++;
      h->host_casts++;
      int st = record_last(h, s);
      if (st != FP8Q_OK) return st;
    }
  }
  return FP8Q_OK;
}

static int check_tensor(fp8q_handle h, const void* x, int dtype, int64_t n, const uint8_t* q) {
  if (!handle_ok(h)) return FP8Q_EHANDLE;
  if (!dtype_ok(dtype)) return FP8Q_EDTYPE;
  if (n < 0 || n > (int64_t(1) << 46)) return FP8Q_EINVAL;
  if (n > 0 && (x == nullptr || q == nullptr)) return FP8Q_EINVAL;
  if (!aligned16(x) || !aligned16(q)) return FP8Q_EALIGN;
  return FP8Q_OK;
}

FP8Q_API int fp8q_cast(fp8q_handle h, const void* x, int dtype, int64_t n, uint8_t* q,
                       float* d_scale_inv, float* d_amax, unsigned long long* d_clipped,
                       void* stream) {
  FP8Q_TRACE_CALL();
  int st = check_tensor(h, x, dtype, n, q);
  if (st != FP8Q_OK) return st;
  st = check_device(h);
  if (st != FP8Q_OK) return st;
  return plan_and_launch(&h, &x, &dtype, &n, &q, d_scale_inv, d_amax, d_clipped, nullptr, nullptr,
                         1, reinterpret_cast<cudaStream_t>(stream));
}

FP8Q_API int fp8q_cast_multi_ex(const fp8q_handle* hs, const void* const* xs, const int* dtypes,
                                const int64_t* ns, uint8_t* const* qs, float* d_scale_inv,
                                float* d_amax, unsigned long long* d_clipped,
                                unsigned long long* d_nonfinite, unsigned long long* d_underflow,
                                int count, void* stream) {
  FP8Q_TRACE_CALL();
  if (count <= 0 || !hs || !xs || !dtypes || !ns || !qs) return FP8Q_EINVAL;
  for (int i = 0; i < count; ++i) {
    int st = check_tensor(hs[i], xs[i], dtypes[i], ns[i], qs[i]);
    if (st != FP8Q_OK) return st;
    st = check_device(hs[i]);
    if (st != FP8Q_OK) return st;
  }
  std::vector<fp8q_handle> sorted(hs, hs + count);
  std::sort(sorted.begin(), sorted.end());
  if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end()) return FP8Q_EINVAL;
  return plan_and_launch(hs, xs, dtypes, ns, qs, d_scale_inv, d_amax, d_clipped, d_nonfinite,
                         d_underflow, count, reinterpret_cast<cudaStream_t>(stream));
}

FP8Q_API int fp8q_cast_multi(const fp8q_handle* hs, const void* const* xs, const int* dtypes,
                             const int64_t* ns, uint8_t* const* qs, float* d_scale_inv,
                             float* d_amax, unsigned long long* d_clipped, int count,
                             void* stream) {
  FP8Q_TRACE_CALL();
  return fp8q_cast_multi_ex(hs, xs, dtypes, ns, qs, d_scale_inv, d_amax, d_clipped, nullptr, nullptr,
                            count, stream);
}

static const uint32_t kScalerMagic = 0x1055CA1Eu;

}  // extern "C"

struct fp8q_loss_scaler_state {
  uint32_t magic;
  int device;
  LossScaleState* dev;
  cudaEvent_t last;
  bool has_last;
};

extern "C" {

FP8Q_API int fp8q_loss_scaler_create(float init_scale, int growth_interval, float min_scale,
                                     float max_scale, fp8q_loss_scaler* out) {
  FP8Q_TRACE_CALL();
  if (!out) return FP8Q_EINVAL;
  *out = nullptr;
  if (!(min_scale > 0.0f) || !(max_scale >= min_scale) || !(init_scale >= min_scale) ||
      !(init_scale <= max_scale) || growth_interval < 1)
    return FP8Q_EINVAL;
  fp8q_loss_scaler_state* ls = new (std::nothrow) fp8q_loss_scaler_state();
  if (!ls) return FP8Q_ENOMEM;
  cudaError_t e = cudaGetDevice(&ls->device);
  if (e != cudaSuccess) { delete ls; return fail_cuda(e); }
  e = cudaMalloc(reinterpret_cast<void**>(&ls->dev), sizeof(LossScaleState));
  if (e != cudaSuccess) { delete ls; return e == cudaErrorMemoryAllocation ? FP8Q_ENOMEM : fail_cuda(e); }
  LossScaleState init;
  std::memset(&init, 0, sizeof init);
  init.scale = init_scale;
  init.min_scale = min_scale;
  init.max_scale = max_scale;
  init.growth_interval = growth_interval;
  e = cudaMemcpy(ls->dev, &init, sizeof init, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ls->last, cudaEventDisableTiming);
  if (e != cudaSuccess) { cudaFree(ls->dev); delete ls; return fail_cuda(e); }
  ls->has_last = false;
  ls->magic = kScalerMagic;
  *out = ls;
  return FP8Q_OK;
}

FP8Q_API int fp8q_loss_scaler_destroy(fp8q_loss_scaler ls) {
  FP8Q_TRACE_CALL();
  if (!ls) return FP8Q_OK;
  if (ls->magic != kScalerMagic) return FP8Q_EHANDLE;
  if (ls->has_last) cudaEventSynchronize(ls->last);
  cudaEventDestroy(ls->last);
  cudaError_t e = cudaFree(ls->dev);
  ls->magic = 0;
  delete ls;
  return e == cudaSuccess ? FP8Q_OK : fail_cuda(e);
}

FP8Q_API int fp8q_loss_scaler_update(fp8q_loss_scaler ls, const unsigned long long* d_nonfinite,
                                     int count, float* d_scale, int* d_skip, void* stream) {
  FP8Q_TRACE_CALL();
  if (!ls || ls->magic != kScalerMagic) return FP8Q_EHANDLE;
  if (count < 0 || (count > 0 && !d_nonfinite)) return FP8Q_EINVAL;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev != ls->device) return FP8Q_EDEVICE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int launches = 0;
  e = launch_loss_scale_update(ls->dev, d_nonfinite, count, d_scale, d_skip, s, &launches);
  g_launches += launches;
  if (e != cudaSuccess) return fail_cuda(e);
  if (stream_capturing(s)) return FP8Q_OK;      // a captured update: the replays are the caller's to wait for
  e = cudaEventRecord(ls->last, s);
  if (e != cudaSuccess) return fail_cuda(e);
  ls->has_last = true;
  return FP8Q_OK;
}

FP8Q_API int fp8q_loss_scaler_read(fp8q_loss_scaler ls, float* scale, int* good_steps) {
  FP8Q_TRACE_CALL();
  if (!ls || ls->magic != kScalerMagic) return FP8Q_EHANDLE;
  if (ls->has_last) {
    cudaError_t e = cudaEventSynchronize(ls->last);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  LossScaleState d;
  cudaError_t e = cudaMemcpy(&d, ls->dev, sizeof d, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(e);
  if (scale) *scale = d.scale;
  if (good_steps) *good_steps = d.good;
  return FP8Q_OK;
}

FP8Q_API int mx_cast_ex(const void* x, int dtype, int64_t rows, int64_t cols, int format,
                        int rule, int headroom_bits, int axis, uint8_t* q, uint8_t* e8m0,
                        unsigned long long* d_clipped, void* stream) {
  FP8Q_TRACE_CALL();
  if (!dtype_ok(dtype) || !format_ok(format)) return FP8Q_EDTYPE;
  if (rule < FP8Q_MX_FLOOR || rule > FP8Q_MX_NEAREST) return FP8Q_EINVAL;
  if (axis != FP8Q_MX_ROWWISE && axis != FP8Q_MX_COLWISE) return FP8Q_EINVAL;
  if (rows < 0 || cols <= 0 || headroom_bits < 0 || headroom_bits > kMaxHeadroom) return FP8Q_EINVAL;
  if (axis == FP8Q_MX_ROWWISE && cols % 32 != 0) return FP8Q_EINVAL;
  if (axis == FP8Q_MX_COLWISE && (rows % 32 != 0 || cols % 16 != 0)) return FP8Q_EINVAL;
  if (rows > 0 && cols > (int64_t(1) << 46) / rows) return FP8Q_EINVAL;
  const int64_t n = rows * cols;
  if (n > 0 && (!x || !q || !e8m0)) return FP8Q_EINVAL;
  if (!aligned16(x) || !aligned16(q)) return FP8Q_EALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (d_clipped) {
    cudaError_t e = cudaMemsetAsync(d_clipped, 0, sizeof(unsigned long long), s);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  if (n == 0) return FP8Q_OK;
  int launches = 0;
  cudaError_t e = axis == FP8Q_MX_ROWWISE
                      ? launch_mx(x, dtype, n, format, headroom_bits, rule, q, e8m0, d_clipped, s, &launches)
                      : launch_mx_colwise(x, dtype, rows, cols, format, headroom_bits, rule, q, e8m0,
                                          d_clipped, s, &launches);
  g_launches += launches;
  return e == cudaSuccess ? FP8Q_OK : fail_cuda(e);
}

FP8Q_API int mx_cast_dual(const void* x, int dtype, int64_t rows, int64_t cols, int format, int rule,
                          int headroom_bits, uint8_t* q_row, uint8_t* e8m0_row, uint8_t* q_colt,
                          uint8_t* e8m0_colt, unsigned long long* d_clipped_row,
                          unsigned long long* d_clipped_col, void* stream) {
  FP8Q_TRACE_CALL();
  if (!dtype_ok(dtype) || !format_ok(format)) return FP8Q_EDTYPE;
  if (rule < FP8Q_MX_FLOOR || rule > FP8Q_MX_NEAREST) return FP8Q_EINVAL;
  if (rows < 0 || cols <= 0 || rows % 32 != 0 || cols % 32 != 0 || headroom_bits < 0 ||
      headroom_bits > kMaxHeadroom)
    return FP8Q_EINVAL;
  if (rows > 0 && cols > (int64_t(1) << 46) / rows) return FP8Q_EINVAL;
  if (rows >= (int64_t(1) << 31) || cols >= (int64_t(1) << 31)) return FP8Q_EINVAL;
  const int64_t n = rows * cols;
  if (n > 0 && (!x || !q_row || !e8m0_row || !q_colt || !e8m0_colt)) return FP8Q_EINVAL;
  if (!aligned16(x) || !aligned16(q_row) || !aligned16(q_colt)) return FP8Q_EALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  for (unsigned long long* c : {d_clipped_row, d_clipped_col}) {
    if (!c) continue;
    cudaError_t e = cudaMemsetAsync(c, 0, sizeof(unsigned long long), s);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  if (n == 0) return FP8Q_OK;
  int launches = 0;
  cudaError_t e = launch_mx_dual(x, dtype, rows, cols, format, rule, headroom_bits, q_row, e8m0_row,
                                 q_colt, e8m0_colt, d_clipped_row, d_clipped_col, s, &launches);
  g_launches += launches;
  return e == cudaSuccess ? FP8Q_OK : fail_cuda(e);
}

FP8Q_API int fp8q_cast_transpose(fp8q_handle h, const void* x, int dtype, int64_t rows, int64_t cols,
                                 uint8_t* q, uint8_t* qt, float* d_scale_inv, float* d_amax,
                                 unsigned long long* d_clipped, void* stream) {
  FP8Q_TRACE_CALL();
  if (!handle_ok(h)) return FP8Q_EHANDLE;
  if (!dtype_ok(dtype)) return FP8Q_EDTYPE;
  if (rows <= 0 || cols <= 0 || rows % 32 != 0 || cols % 32 != 0) return FP8Q_EINVAL;
  if (cols > (int64_t(1) << 46) / rows || rows >= (int64_t(1) << 31) || cols >= (int64_t(1) << 31))
    return FP8Q_EINVAL;
  if (!x || !q || !qt) return FP8Q_EINVAL;
  if (!aligned16(x) || !aligned16(q) || !aligned16(qt)) return FP8Q_EALIGN;
  int st = check_device(h);
  if (st != FP8Q_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (stream_capturing(s) && first_windowed_cast(h)) return FP8Q_EINVAL;
  const int64_t n = rows * cols;
  const bool current = h->estimator == FP8Q_EST_SMOOTHED ? h->host_casts == 0
                                                         : (h->window == 0 || h->host_count == 0);
  int launches = 0;
  GroupHeader gh;
  std::memset(&gh, 0, sizeof gh);
  if (current) {
    const int64_t ce = chunk_elems(dtype);
    const long long nch = (n + ce - 1) / ce;
    if (nch > 0x7FFFFFFFll) return FP8Q_EINVAL;
    TensorDesc d;
    d.x = x;
    d.q = q;
    d.n = n;
    d.st = h->dev;
    d.chunk_begin = 0;
    d.flags = (dtype == FP8Q_BF16 ? 1 : 0) | (h->format == FP8Q_E5M2 ? 2 : 0) | (kCurrentPre << 2);
    gh.total_chunks = (int32_t)nch;
    cudaError_t e = launch_amax_group(gh, &d, 1, s, &launches);
    g_launches += launches;
    launches = 0;
    if (e != cudaSuccess) return fail_cuda(e);
  }
  gh.scale_inv = d_scale_inv;
  gh.amax = d_amax;
  gh.clipped = d_clipped;
  gh.count = 1;
  cudaError_t e = launch_cast_transpose(x, dtype, h->format, rows, cols, q, qt, h->dev,
                                        current ? kCurrentPre : kDelayed, gh, s, &launches);
  g_launches += launches;
  if (e != cudaSuccess) return fail_cuda(e);
  if (h->window > 0 && h->host_count < h->window) h->host_count++;
  h->host_casts++;
  return record_last(h, s);
}

FP8Q_API int mx_cast(const void* x, int dtype, int64_t rows, int64_t cols, int format,
                     int headroom_bits, uint8_t* q, uint8_t* e8m0,
                     unsigned long long* d_clipped, void* stream) {
  FP8Q_TRACE_CALL();
  return mx_cast_ex(x, dtype, rows, cols, format, FP8Q_MX_FLOOR, headroom_bits, FP8Q_MX_ROWWISE,
                    q, e8m0, d_clipped, stream);
}

FP8Q_API int fp8q_amax_history(fp8q_handle h, float* host_out, int capacity, int* n_valid) {
  FP8Q_TRACE_CALL();
  if (!handle_ok(h)) return FP8Q_EHANDLE;
  if (!n_valid || (capacity > 0 && !host_out) || capacity < h->window) return FP8Q_EINVAL;
  int st = check_device(h);
  if (st == FP8Q_OK) st = wait_last(h);
  if (st != FP8Q_OK) return st;
  DevState d;
  cudaError_t e = cudaMemcpy(&d, h->dev, sizeof d, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(e);
  const int cnt = d.count;
  // oldest first: with a full ring the oldest entry sits at head
  for (int i = 0; i < cnt; ++i) {
    const int slot = (cnt < h->window) ? i : (d.head + i) % h->window;
    std::memcpy(&host_out[i], &d.ring[slot], 4);
  }
  *n_valid = cnt;
  return FP8Q_OK;
}

FP8Q_API int fp8q_scale_state(fp8q_handle h, int* prev_exp, long long* steps) {
  FP8Q_TRACE_CALL();
  if (!handle_ok(h)) return FP8Q_EHANDLE;
  int st = check_device(h);
  if (st == FP8Q_OK) st = wait_last(h);
  if (st != FP8Q_OK) return st;
  DevState d;
  cudaError_t e = cudaMemcpy(&d, h->dev, sizeof d, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(e);
  if (prev_exp) *prev_exp = d.has_prev ? d.prev_e : FP8Q_NO_EXP;
  if (steps) *steps = d.steps;
  return FP8Q_OK;
}

// Write a handle's window (n values, oldest first) and previous exponent.
// keep_estimator: the running average, the number of casts and the interval
// phase are read back and kept (a restore of the window alone); otherwise
// they are cleared with everything else (a reset).
static int write_state(fp8q_handle h, const float* host_in, int n, int prev_exp, bool keep_estimator) {
  int st = check_device(h);
  if (st == FP8Q_OK) st = wait_last(h);
  if (st != FP8Q_OK) return st;
  DevState old;
  std::memset(&old, 0, sizeof old);
  if (keep_estimator) {
    cudaError_t e = cudaMemcpy(&old, h->dev, sizeof old, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  DevState d;
  std::memset(&d, 0, sizeof d);
  d.format = h->format;
  d.window = h->window;
  d.margin = h->margin;
  d.hyst = h->hyst;
  d.estimator = h->estimator;
  d.alpha = h->alpha;
  d.interval = h->interval;
  for (int i = 0; i < n; ++i) {
    uint32_t b;
    std::memcpy(&b, &host_in[i], 4);
    b &= 0x7FFFFFFFu;
    d.ring[i] = b > 0x7F800000u ? 0x7FC00000u : b;
  }
  d.count = n;
  d.head = (h->window > 0) ? n % h->window : 0;
  d.has_prev = prev_exp != FP8Q_NO_EXP;
  d.prev_e = d.has_prev ? prev_exp : 0;
  d.steps = old.steps;
  d.phase = old.phase;
  d.avg = old.avg;
  d.has_avg = old.has_avg;
  cudaError_t e = cudaMemcpy(h->dev, &d, sizeof d, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return fail_cuda(e);
  h->host_count = n;
  h->host_casts = d.steps;
  return FP8Q_OK;
}

FP8Q_API int fp8q_get_estimator_state(fp8q_handle h, float* average, int* has_average,
                                      long long* steps) {
  FP8Q_TRACE_CALL();
  if (!handle_ok(h)) return FP8Q_EHANDLE;
  int st = check_device(h);
  if (st == FP8Q_OK) st = wait_last(h);
  if (st != FP8Q_OK) return st;
  DevState d;
  cudaError_t e = cudaMemcpy(&d, h->dev, sizeof d, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(e);
  if (average) *average = d.avg;
  if (has_average) *has_average = d.has_avg;
  if (steps) *steps = d.steps;
  return FP8Q_OK;
}

FP8Q_API int fp8q_set_estimator_state(fp8q_handle h, float average, int has_average,
                                      long long steps) {
  FP8Q_TRACE_CALL();
  if (!handle_ok(h)) return FP8Q_EHANDLE;
  if (steps < 0) return FP8Q_EINVAL;
  int st = check_device(h);
  if (st == FP8Q_OK) st = wait_last(h);
  if (st != FP8Q_OK) return st;
  DevState d;
  cudaError_t e = cudaMemcpy(&d, h->dev, sizeof d, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(e);
  d.avg = average;
  d.has_avg = has_average ? 1 : 0;
  d.steps = steps;
  d.phase = (int32_t)(steps % h->interval);
  e = cudaMemcpy(h->dev, &d, sizeof d, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return fail_cuda(e);
  h->host_casts = steps;
  return FP8Q_OK;
}

FP8Q_API int fp8q_set_history(fp8q_handle h, const float* host_in, int n, int prev_exp) {
  FP8Q_TRACE_CALL();
  if (!handle_ok(h)) return FP8Q_EHANDLE;
  if (n < 0 || n > h->window || (n > 0 && !host_in)) return FP8Q_EINVAL;
  if (prev_exp != FP8Q_NO_EXP && (prev_exp < -126 || prev_exp > 126)) return FP8Q_EINVAL;
  return write_state(h, host_in, n, prev_exp, true);
}

FP8Q_API int fp8q_reset(fp8q_handle h) {
  FP8Q_TRACE_CALL();
  if (!handle_ok(h)) return FP8Q_EHANDLE;
  return write_state(h, nullptr, 0, FP8Q_NO_EXP, false);
}

FP8Q_API int fp8q_error_stats(const void* x, int dtype, int64_t n, const uint8_t* q, int format,
                              const float* d_scale_inv, double* d_out, void* stream) {
  FP8Q_TRACE_CALL();
  if (!dtype_ok(dtype) || !format_ok(format)) return FP8Q_EDTYPE;
  if (n < 0 || !d_out || !d_scale_inv || (n > 0 && (!x || !q))) return FP8Q_EINVAL;
  int launches = 0;
  cudaError_t e = launch_stats(x, dtype, n, q, format, d_scale_inv, nullptr, d_out,
                               reinterpret_cast<cudaStream_t>(stream), &launches);
  g_launches += launches;
  return e == cudaSuccess ? FP8Q_OK : fail_cuda(e);
}

FP8Q_API int mx_error_stats(const void* x, int dtype, int64_t rows, int64_t cols,
                            const uint8_t* q, const uint8_t* e8m0, int format, double* d_out,
                            void* stream) {
  FP8Q_TRACE_CALL();
  if (!dtype_ok(dtype) || !format_ok(format)) return FP8Q_EDTYPE;
  if (rows < 0 || cols <= 0 || cols % 32 != 0 || !d_out) return FP8Q_EINVAL;
  const int64_t n = rows * cols;
  if (n > 0 && (!x || !q || !e8m0)) return FP8Q_EINVAL;
  int launches = 0;
  cudaError_t e = launch_stats(x, dtype, n, q, format, nullptr, e8m0, d_out,
                               reinterpret_cast<cudaStream_t>(stream), &launches);
  g_launches += launches;
  return e == cudaSuccess ? FP8Q_OK : fail_cuda(e);
}

}  // extern "C"

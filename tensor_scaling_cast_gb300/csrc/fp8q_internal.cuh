// Internal definitions shared by the libfp8q translation units (device
// state layout, launch descriptors, small device helpers).
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "fp8q.h"

namespace fp8q {

// NVTX range over one C-ABI call, named after the entry point, in the
// library's own "fp8q" domain.  With no tool attached NVTX's entry points
// return at once, so the range costs a call and a branch.
inline nvtxDomainHandle_t trace_domain() {
  static const nvtxDomainHandle_t d = nvtxDomainCreateA("fp8q");
  return d;
}
struct TraceRange {
  explicit TraceRange(const char* name) {
    nvtxEventAttributes_t a = {};
    a.version = NVTX_VERSION;
    a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
    a.messageType = NVTX_MESSAGE_TYPE_ASCII;
    a.message.ascii = name;
    nvtxDomainRangePushEx(trace_domain(), &a);
  }
  ~TraceRange() { nvtxDomainRangePop(trace_domain()); }
  TraceRange(const TraceRange&) = delete;
  TraceRange& operator=(const TraceRange&) = delete;
};
#define FP8Q_TRACE_CALL() ::fp8q::TraceRange fp8q_trace_range_(__func__)

constexpr int kThreads = 256;                 // threads per CTA (8 warps)
constexpr int kUnroll = 8;                    // 16-byte loads in flight per thread
constexpr int kChunkBytes = kThreads * kUnroll * 16;   // 32 KiB of input per chunk
constexpr int kMaxGroup = 512;                // tensors per grouped launch

// Device-resident scaling state of one tensor (one per handle).
struct __align__(256) DevState {
  uint32_t ring[FP8Q_MAX_WINDOW];   // amax fp32 bits of past casts (ring order)
  uint32_t amax_acc;                // running max of |x| bits, this cast
  uint32_t pre_amax;                // current-scaling pre-pass result
  unsigned long long clip_acc;      // clipped elements, this cast
  unsigned long long nonfinite_acc; // NaN / Inf inputs, this cast
  unsigned long long underflow_acc; // finite nonzero inputs cast to zero, this cast
  uint32_t ticket;                  // chunks finished, this cast
  int32_t count;                    // valid ring entries (<= window)
  int32_t head;                     // next ring slot
  int32_t prev_e;                   // exponent of the last cast
  int32_t has_prev;
  int32_t format, window, margin, hyst;
  long long steps;                  // casts done
  int32_t estimator;                // FP8Q_EST_MAX_WINDOW or FP8Q_EST_SMOOTHED
  float alpha;                      // smoothing coefficient
  int32_t interval;                 // recompute the exponent every `interval` casts
  int32_t phase;                    // casts done, modulo interval
  float avg;                        // running average of the amax (smoothed estimator)
  int32_t has_avg;
};

enum Mode : int { kDelayed = 0, kCurrentPre = 1, kCurrentLocal = 2 };

// One tensor of a grouped launch (40 bytes; kept in the kernel's
// parameter space, so a 512-tensor group needs no device-side table).
struct TensorDesc {
  const void* x;
  uint8_t* q;
  int64_t n;
  DevState* st;
  int32_t chunk_begin;              // first chunk of this tensor in the group
  int32_t flags;                    // bit0 bf16, bit1 E5M2, bits2-3 Mode
};

struct GroupHeader {
  float* scale_inv;                 // [out_offset + t] outputs, nullable
  float* amax;
  unsigned long long* clipped;
  unsigned long long* nonfinite;
  unsigned long long* underflow;    // non-null: the underflow-counting kernel runs
  int32_t count;
  int32_t total_chunks;
  int32_t out_offset;
  int32_t pad;
};

template <int MAXT>
struct GroupParams {
  GroupHeader h;
  TensorDesc d[MAXT];
};

inline int chunk_elems(int dtype) { return kChunkBytes / (dtype == FP8Q_BF16 ? 2 : 4); }

// ---- launches (defined in cast.cu / mx.cu / stats.cu) ----------------------
// Each returns a cudaError_t from the launch.
cudaError_t launch_cast_group(const GroupHeader& h, const TensorDesc* d, int count,
                              cudaStream_t s, int* launches);
cudaError_t launch_amax_group(const GroupHeader& h, const TensorDesc* d, int count,
                              cudaStream_t s, int* launches);
cudaError_t launch_mx(const void* x, int dtype, int64_t nelem, int format, int headroom, int rule,
                      uint8_t* q, uint8_t* e8m0, unsigned long long* clipped, cudaStream_t s,
                      int* launches);
cudaError_t launch_mx_colwise(const void* x, int dtype, int64_t rows, int64_t cols, int format,
                              int headroom, int rule, uint8_t* q, uint8_t* e8m0,
                              unsigned long long* clipped, cudaStream_t s, int* launches);
cudaError_t launch_stats(const void* x, int dtype, int64_t n, const uint8_t* q, int format,
                         const float* scale_inv, const uint8_t* e8m0, double* out,
                         cudaStream_t s, int* launches);

cudaError_t read_wait_timeouts(unsigned int* count);      // and reset to 0 (mx.cu)
cudaError_t launch_pipeline_selftest(cudaStream_t s, int* launches);
cudaError_t launch_warp_pipe_selftest(cudaStream_t s, int* launches);   // transpose.cu
cudaError_t read_tp_wait_timeouts(unsigned int* count);   // and reset to 0 (transpose.cu)
cudaError_t launch_mx_dual(const void* x, int dtype, int64_t rows, int64_t cols, int format, int rule,
                           int headroom, uint8_t* q_row, uint8_t* e8_row, uint8_t* q_colt,
                           uint8_t* e8_colt, unsigned long long* cr, unsigned long long* cc,
                           cudaStream_t s, int* launches);
cudaError_t launch_cast_transpose(const void* x, int dtype, int format, int64_t rows, int64_t cols,
                                  uint8_t* q, uint8_t* qt, DevState* st, int mode, const GroupHeader& h,
                                  cudaStream_t s, int* launches);

// Device state of a dynamic loss scaler.
struct LossScaleState {
  float scale, min_scale, max_scale;
  int32_t growth_interval, good, last_skip;
  long long updates;
};
cudaError_t launch_loss_scale_update(LossScaleState* st, const unsigned long long* nonfinite, int count,
                                     float* scale_out, int* skip_out, cudaStream_t s, int* launches);

int sm_count(int device);
cudaError_t kernel_occupancy(const void* kernel, int threads, int smem, int* occ);
int record_cuda_error(cudaError_t e);   // keeps the text, returns FP8Q_ECUDA
void note_launches(int k);              // adds to fp8q_launch_count()
int device_of_current();

}  // namespace fp8q

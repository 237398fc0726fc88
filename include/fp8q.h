/*
 * fp8q.h -- C ABI of libfp8q, a GB300 (sm_103a) library for the scaled cast
 * of training tensors to 8-bit floats.
 *
 * What it computes, and where the pages define it:
 *  - Formats ("Mixed Precision FP16/BF16/FP8" mind-map card, bit layouts and
 *    ranges, item 3): OCP E4M3 (4 exponent + 3 mantissa bits, largest finite
 *    448) for weights and activations, OCP E5M2 (5 + 2, largest finite 57344)
 *    for gradients.
 *  - Per-tensor scale ("Practice c06/E3", worked solution): watch the largest
 *    |x| of a tensor over a window of steps; the scale is the largest power
 *    of two keeping that value at or below the format's largest finite value
 *    divided by 2^margin; keep the previous scale under a hysteresis rule.
 *  - Window variants (gist.science summary of "Max-Window Scale Estimation
 *    for Near-Lossless HiF8 W8A8 QAT", Methodology, "Amax algorithms"):
 *    most-recent (window 1), max over a history window, current tensor
 *    scaling (window 0 here).
 *  - MX block scaling ("what actually breaks low precision training", "What
 *    the measurements said"): one shared power of two per 32 values from the
 *    OCP formula floor(log2(block amax)) - emax_elem; one extra bit of
 *    exponent headroom as an option.
 *
 * Semantics fixed by this library where the pages are silent:
 *  - Rounding: round to nearest, ties to even, on the format's grid; a
 *    magnitude that rounds past the largest finite value saturates to
 *    sign|max and counts as clipped (E4M3: |v| > 464; E5M2: |v| >= 61440).
 *    +-Inf inputs saturate and count as clipped.  NaN -> sign|0x7F, not
 *    clipped.  Zero and values that round to zero keep their sign.
 *  - amax: max |x| with NaN > Inf > finite; any NaN gives the canonical NaN.
 *  - Scale exponent e (scale = 2^e, scale_inv = 2^-e) is clamped to
 *    [-126, 126].  A zero or non-finite window maximum keeps the previous e
 *    (0 if none).  Hysteresis h: an upward move of 1..h binades keeps the
 *    previous e; downward moves are immediate.
 *  - The window holds the amaxes of the previous `window` casts of the
 *    handle; the current amax enters it after the cast.  An empty window
 *    (first cast, or window 0) uses current scaling: amax of this tensor
 *    first, then the cast (two reads of x).
 *  - MX: E clamped to [-127, 127]; an all-zero block gets E = -127 (byte
 *    0x00); a block holding NaN or Inf gets E8M0 0xFF and every element byte
 *    sign|0x7F.
 *
 * Conventions for every call:
 *  - Return value: FP8Q_OK (0) or a negative FP8Q_E* status.  Nothing
 *    throws.  fp8q_strerror() names a status; fp8q_last_cuda_error() gives
 *    the text of the last CUDA error seen by the calling thread.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls taking a stream only enqueue work and return; outputs
 *    are device memory, valid once the stream reaches that point.
 *  - Tensors (x, q, e8m0, outputs) are device pointers owned by the caller;
 *    the library never frees or retains them.  x and q must be 16-byte
 *    aligned (else FP8Q_EALIGN).  x is read as a contiguous 1-D array of n
 *    elements; q receives n bytes in the same order.
 *  - A handle belongs to the device that was current at fp8q_create and must
 *    be used with that device current (else FP8Q_EDEVICE).  A handle keeps
 *    state across calls: do not use one handle from two streams or two host
 *    threads at once.  Distinct handles are independent: casts on different
 *    handles may run on different streams and host threads concurrently.
 *  - The library has no CPU path: without a usable GPU every compute call
 *    returns FP8Q_ECUDA.
 */
#ifndef FP8Q_H
#define FP8Q_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define FP8Q_API __attribute__((visibility("default")))
#else
#define FP8Q_API
#endif

/* 8-bit target formats */
enum { FP8Q_E4M3 = 0, FP8Q_E5M2 = 1 };
/* input element types */
enum { FP8Q_F32 = 0, FP8Q_BF16 = 1 };
/* status codes */
enum {
  FP8Q_OK = 0,
  FP8Q_EINVAL = -1,   /* bad argument value (size, window, null pointer, ...) */
  FP8Q_EALIGN = -2,   /* x or q not 16-byte aligned                         */
  FP8Q_EDTYPE = -3,   /* unknown dtype or format                            */
  FP8Q_ECUDA = -4,    /* a CUDA call failed; see fp8q_last_cuda_error()     */
  FP8Q_EHANDLE = -5,  /* null or destroyed handle                           */
  FP8Q_ENOMEM = -6,   /* device or host allocation failed                   */
  FP8Q_EDEVICE = -7,  /* handle used with another device current            */
  FP8Q_ESIZE = -8     /* size above the limit of a fixed-size scratch area  */
};

/* Largest history window a handle may keep. */
#define FP8Q_MAX_WINDOW 256
/* "No previous exponent" in fp8q_scale_state / fp8q_set_history. */
#define FP8Q_NO_EXP (-2147483647 - 1)

typedef struct fp8q_state* fp8q_handle;

/* Create the scaling state of one tensor ("Practice c06/E3" worked solution:
 * per-tensor statistic, window, margin, hysteresis).
 *   format      FP8Q_E4M3 or FP8Q_E5M2
 *   window      0 (current scaling every call) .. FP8Q_MAX_WINDOW
 *   margin_bits >= 0 and <= 16: the scale keeps amax <= fmax / 2^margin
 *   hysteresis_bits >= 0 and <= 16 (0 = off)
 * Allocates the state in device memory of the current device (cudaMalloc).
 * *out receives the handle; FP8Q_ENOMEM / FP8Q_ECUDA on failure.  The state
 * lives in the device's current context: once that context is destroyed
 * (cudaDeviceReset), destroy the handle and create a new one -- the old
 * handle's device state no longer exists. */
FP8Q_API int fp8q_create(int format, int window, int margin_bits, int hysteresis_bits,
                         fp8q_handle* out);

/* Estimators of the statistic the scale comes from (gist.science summary of
 * "Max-Window Scale Estimation ...", Methodology, "Amax algorithms"):
 *   FP8Q_EST_MAX_WINDOW  the largest amax of the last `window` casts (window 1
 *                        is the most-recent rule, window 0 current scaling)
 *   FP8Q_EST_SMOOTHED    a running average of the amax ("exponential
 *                        smoothing", coefficient not given by the pages):
 *                        avg <- avg + alpha * (amax - avg) in fp32 (three
 *                        roundings, no FMA), started at the first cast's amax;
 *                        a non-finite amax does not enter the average. */
enum { FP8Q_EST_MAX_WINDOW = 0, FP8Q_EST_SMOOTHED = 1 };

/* fp8q_create with a choice of estimator and a recompute interval
 * ("Practice c06/E3" worked solution: recompute the scale every fixed number
 * of steps).
 *   estimator  FP8Q_EST_MAX_WINDOW or FP8Q_EST_SMOOTHED
 *   alpha      smoothing coefficient in (0, 1] (used by FP8Q_EST_SMOOTHED)
 *   interval   >= 1: the exponent is recomputed only when the number of
 *              earlier casts is a multiple of interval, and kept otherwise
 * With FP8Q_EST_SMOOTHED the window only sizes the history that
 * fp8q_amax_history reports; the first cast uses current scaling. */
FP8Q_API int fp8q_create_ex(int format, int window, int margin_bits, int hysteresis_bits,
                            int estimator, float alpha, int interval, fp8q_handle* out);

/* Read / restore the estimator state that fp8q_set_history does not cover:
 * the running average (valid when *has_average) and the number of casts
 * done (the phase of the recompute interval).  Setting it leaves the window
 * and the previous exponent as they are.  Both block until the handle's
 * last cast has finished. */
FP8Q_API int fp8q_get_estimator_state(fp8q_handle h, float* average, int* has_average,
                                      long long* steps);
FP8Q_API int fp8q_set_estimator_state(fp8q_handle h, float average, int has_average,
                                      long long steps);

/* Free a handle's device and host state.  Waits for the handle's last cast.
 * NULL is accepted (returns FP8Q_OK). */
FP8Q_API int fp8q_destroy(fp8q_handle h);

/* Fused scaled cast of one tensor ("Practice c06/E3", worked solution: the
 * largest |x| of the tensor watched over a window of steps sets a
 * power-of-two scale; "Mixed Precision FP16/BF16/FP8" mind-map card, bit
 * layouts and ranges: E4M3 max 448, E5M2 max 57344; gist.science summary of
 * "Max-Window Scale Estimation ...", Methodology: the delayed estimators use
 * historical amaxes, current scaling a second pass).  Steps: amax reduction,
 * scale from the window, saturating RNE cast with clipped count, cross-CTA
 * finish.
 *   x       device, n elements of `dtype` (FP8Q_F32 or FP8Q_BF16), 16-B aligned
 *   n       >= 0 elements (any n; n = 0 records amax 0)
 *   q       device, n bytes out (the handle's format), 16-B aligned
 *   d_scale_inv, d_amax  device float out (scale_inv = 2^-e; amax of x), or NULL
 *   d_clipped            device uint64 out (clipped count), or NULL
 * One launch with a non-empty window (each element read once); two launches
 * for current scaling of a tensor larger than one CTA chunk. */
FP8Q_API int fp8q_cast(fp8q_handle h, const void* x, int dtype, int64_t n, uint8_t* q,
                       float* d_scale_inv, float* d_amax, unsigned long long* d_clipped,
                       void* stream);

/* Grouped version of fp8q_cast over `count` tensors in one launch (plus one
 * amax pre-pass launch if any tensor needs current scaling).  Each tensor
 * keeps its own statistic and scale ("Practice c06/E3", worked solution:
 * the scale is set per tensor rather than per run; gist.science summary of
 * "Max-Window Scale Estimation ...", Methodology, Quantization
 * Configuration: W8A8 casts the weights and the activations of the gate, up
 * and down projections of many blocks at every step).  hs, xs,
 * dtypes, ns, qs are HOST arrays of length count (xs/qs hold device
 * pointers); the handles must be distinct.  d_scale_inv, d_amax, d_clipped
 * are DEVICE arrays of length count (or NULL).  Work is split into equal
 * 32 KiB input chunks over all tensors; each tensor keeps its own state.
 * count > 0; groups above 512 tensors are split into several launches.
 *
 * CUDA graphs (stream capture), for fp8q_cast, fp8q_cast_multi(_ex),
 * fp8q_cast_transpose and fp8q_loss_scaler_update: a cast may be captured
 * once each of its handles has done its first cast, or has window 0 under
 * the max-window estimator.  A handle's first cast under a window or the
 * smoothed estimator takes the current-scaling path, chosen on the host, so
 * while its stream captures it returns FP8Q_EINVAL and captures nothing.
 * Every launch of the graph advances the handles' device state exactly as
 * the same eager calls would.  A captured call does not mark its handle:
 * synchronise the stream the graph runs on before reading or setting the
 * handle's state (fp8q_amax_history, fp8q_scale_state, fp8q_set_history,
 * fp8q_reset, the estimator state, fp8q_loss_scaler_read), which are host
 * calls and not capturable themselves. */
FP8Q_API int fp8q_cast_multi(const fp8q_handle* hs, const void* const* xs, const int* dtypes,
                             const int64_t* ns, uint8_t* const* qs, float* d_scale_inv,
                             float* d_amax, unsigned long long* d_clipped, int count,
                             void* stream);

/* fp8q_cast_multi with two more per-tensor counts (DEVICE arrays of length
 * count, or NULL):
 *   d_nonfinite  NaN or +-Inf inputs ("Mixed Precision FP16/BF16/FP8": the
 *                Inf/NaN detection that dynamic loss scaling reacts to)
 *   d_underflow  finite nonzero inputs whose 8-bit result is a zero ("what
 *                actually breaks low precision training": underflow rates)
 * Counting underflow adds work to every element; with d_underflow NULL the
 * launch is the same as fp8q_cast_multi's.  Non-finite inputs are counted on
 * the path that already handles them, at no cost otherwise. */
FP8Q_API int fp8q_cast_multi_ex(const fp8q_handle* hs, const void* const* xs, const int* dtypes,
                                const int64_t* ns, uint8_t* const* qs, float* d_scale_inv,
                                float* d_amax, unsigned long long* d_clipped,
                                unsigned long long* d_nonfinite, unsigned long long* d_underflow,
                                int count, void* stream);

/* Dynamic loss scaling, device-resident ("Mixed Precision FP16/BF16/FP8"
 * mind-map card: multiply the loss by S, commonly 2^24 or 1024; on Inf/NaN
 * set S <- S/2 and skip the step; after a period without overflow double S).
 * The period is growth_interval clean steps in a row; S stays within
 * [min_scale, max_scale].  Allocates its state with cudaMalloc. */
typedef struct fp8q_loss_scaler_state* fp8q_loss_scaler;
FP8Q_API int fp8q_loss_scaler_create(float init_scale, int growth_interval, float min_scale,
                                     float max_scale, fp8q_loss_scaler* out);
FP8Q_API int fp8q_loss_scaler_destroy(fp8q_loss_scaler ls);
/* One step: d_nonfinite is a DEVICE array of `count` non-finite counts (as
 * written by fp8q_cast_multi_ex for the step's gradient casts); the step is
 * non-finite when any is nonzero.  Writes the new scale to *d_scale and 1
 * (skip the step) or 0 to *d_skip (device pointers, either may be NULL).
 * One single-CTA launch. */
FP8Q_API int fp8q_loss_scaler_update(fp8q_loss_scaler ls, const unsigned long long* d_nonfinite,
                                     int count, float* d_scale, int* d_skip, void* stream);
/* Current scale and clean-step streak; blocks until the last update ran. */
FP8Q_API int fp8q_loss_scaler_read(fp8q_loss_scaler ls, float* scale, int* good_steps);

/* MX block-scaled cast ("what actually breaks low precision training", "What
 * the measurements said"): x is a row-major [rows, cols] tensor; each 32
 * consecutive elements of a row share E = floor(log2(block amax)) -
 * emax_elem + headroom_bits (emax_elem 8 for E4M3, 15 for E5M2).
 *   cols          > 0 and a multiple of 32 (else FP8Q_EINVAL)
 *   headroom_bits 0 (OCP rule) .. 4
 *   q             device [rows, cols] bytes; e8m0: device [rows, cols/32] bytes (E+127)
 *   d_clipped     device uint64 out (clipped elements), or NULL
 * One kernel launch (plus a memset of d_clipped). */
FP8Q_API int mx_cast(const void* x, int dtype, int64_t rows, int64_t cols, int format,
                     int headroom_bits, uint8_t* q, uint8_t* e8m0,
                     unsigned long long* d_clipped, void* stream);

/* MX scale-rounding rules and block directions for mx_cast_ex.  The pages
 * ("what actually breaks low precision training", "The part I would rather
 * not write") name the OCP floor rule, NVIDIA's MXFP8 recipe that rounds the
 * shared scale up, and a comparison of floor, ceil and nearest rounding.
 *   FP8Q_MX_FLOOR    E = floor(log2 A) - emax_elem (the OCP formula)
 *   FP8Q_MX_CEIL     the smallest E with A * 2^-E <= fmax (never clips the block max)
 *   FP8Q_MX_NEAREST  the integer E nearest to log2(A / fmax)
 *   FP8Q_MX_ROWWISE  blocks of 32 consecutive elements of a row; e8m0 [rows, cols/32]
 *   FP8Q_MX_COLWISE  blocks of 32 consecutive rows of a column; e8m0 [rows/32, cols] */
enum { FP8Q_MX_FLOOR = 0, FP8Q_MX_CEIL = 1, FP8Q_MX_NEAREST = 2 };
enum { FP8Q_MX_ROWWISE = 0, FP8Q_MX_COLWISE = 1 };

/* MX cast with a choice of rule and block direction (mx_cast is the
 * FP8Q_MX_FLOOR / FP8Q_MX_ROWWISE case).  E += headroom_bits (0..4), then
 * clamped to [-127, 127].  q is row-major [rows, cols] in both directions.
 *   rowwise: cols a multiple of 32.
 *   colwise: rows a multiple of 32, cols a multiple of 16.
 * One kernel launch (plus a memset of d_clipped). */
FP8Q_API int mx_cast_ex(const void* x, int dtype, int64_t rows, int64_t cols, int format,
                        int rule, int headroom_bits, int axis, uint8_t* q, uint8_t* e8m0,
                        unsigned long long* d_clipped, void* stream);

/* Fused cast + transpose of a row-major [rows, cols] tensor with the
 * handle's per-tensor scale: q [rows, cols] and its transpose qt [cols, rows]
 * from one read of x, for matmuls that need both operands cast ("what
 * actually breaks low precision training": real low-precision training casts
 * both operands of the backward matmuls).  Scale, amax, clipped count and
 * the history update are those of fp8q_cast on the same data (clipped
 * elements are counted once).  rows and cols multiples of 32; x, q, qt
 * 16-byte aligned.  One launch (plus the amax pre-pass under current
 * scaling). */
FP8Q_API int fp8q_cast_transpose(fp8q_handle h, const void* x, int dtype, int64_t rows, int64_t cols,
                                 uint8_t* q, uint8_t* qt, float* d_scale_inv, float* d_amax,
                                 unsigned long long* d_clipped, void* stream);

/* MX dual cast: from one read of x [rows, cols], the row-wise MX cast
 * (q_row [rows, cols], e8m0_row [rows, cols/32]) and the column-wise one
 * written transposed, i.e. the row-wise MX cast of x^T (q_colt [cols, rows],
 * e8m0_colt [cols, rows/32]).  Rule and headroom as mx_cast_ex.  rows and
 * cols multiples of 32; x, q_row, q_colt 16-byte aligned.  d_clipped_row /
 * d_clipped_col: device uint64 or NULL.  One launch (plus memsets). */
FP8Q_API int mx_cast_dual(const void* x, int dtype, int64_t rows, int64_t cols, int format, int rule,
                          int headroom_bits, uint8_t* q_row, uint8_t* e8m0_row, uint8_t* q_colt,
                          uint8_t* e8m0_colt, unsigned long long* d_clipped_row,
                          unsigned long long* d_clipped_col, void* stream);

/* Read a handle's amax history (oldest first) to host memory ("Practice
 * c06/E3", worked solution: the window of past largest |x| values the scale
 * comes from; gist.science summary of "Max-Window Scale Estimation ...",
 * Methodology: the history is filled during a BF16 warm-up, so it is
 * training state worth saving).  Blocks until the handle's last cast has
 * finished.  capacity must be >= the window;
 * *n_valid receives the number of entries written. */
FP8Q_API int fp8q_amax_history(fp8q_handle h, float* host_out, int capacity, int* n_valid);

/* Read the exponent chosen by the last cast (FP8Q_NO_EXP if none yet) and
 * the number of casts done.  Blocks like fp8q_amax_history.  Either
 * pointer may be NULL. */
FP8Q_API int fp8q_scale_state(fp8q_handle h, int* prev_exp, long long* steps);

/* Restore a handle's window (resume from a checkpoint; "Practice c06/E3",
 * worked solution: the window and the previous scale that hysteresis keeps;
 * gist.science summary of "Max-Window Scale Estimation ...", Methodology: a
 * history filled before quantising): n (<= window) amax values, oldest
 * first, and the previous exponent (FP8Q_NO_EXP for none).  Only the window
 * and the previous exponent change: the estimator state of
 * fp8q_set_estimator_state (running average, number of casts, interval
 * phase) is kept, so the two restores may come in either order.  Blocks
 * until the handle's last cast has finished. */
FP8Q_API int fp8q_set_history(fp8q_handle h, const float* host_in, int n, int prev_exp);

/* Clear a handle's history, previous exponent and estimator state (as after
 * fp8q_create). */
FP8Q_API int fp8q_reset(fp8q_handle h);

/* Dequantised-error statistics of a per-tensor cast, over the elements whose
 * input is finite ("what actually breaks low precision training": error size
 * and bias measured separately).  deq = decode(q) * (*d_scale_inv).
 *   d_out  device double[3] out: mean squared error, mean error (bias), count
 * Sums are fp64, reduced in a fixed order (deterministic for a given GPU).
 * Uses stream-ordered temporary device memory (cudaMallocAsync). */
FP8Q_API int fp8q_error_stats(const void* x, int dtype, int64_t n, const uint8_t* q, int format,
                              const float* d_scale_inv, double* d_out, void* stream);

/* Same for an MX cast: deq = decode(q) * 2^E of its block; blocks whose
 * E8M0 byte is 0xFF (NaN) are skipped. */
FP8Q_API int mx_error_stats(const void* x, int dtype, int64_t rows, int64_t cols,
                            const uint8_t* q, const uint8_t* e8m0, int format, double* d_out,
                            void* stream);

/* Allocation-free variant of fp8q_error_stats (this entry point has no
 * counterpart on the pages; it exists for callers of this library that
 * cannot allocate device memory).  Some callers cannot call cudaMalloc or
 * cudaMallocAsync at the point where they want the statistics: a framework
 * whose caching allocator already owns all of the device's memory (an extra
 * allocation fails or forces the pool to give memory back), a diagnostic
 * that runs right after an out-of-memory error, or a latency-bound loop in
 * which an allocation may synchronize the device.  fp8q_error_stats
 * allocates its per-CTA partial sums with cudaMallocAsync; this entry point
 * takes them from a fixed array in the library's device memory instead and
 * calls no allocating routine.
 *   Arguments, outputs and results: as fp8q_error_stats (the fp64 sums are
 *   added in a different order, so results may differ in the last bits).
 *   n must be <= FP8Q_STATS_NOALLOC_MAX_N, else FP8Q_ESIZE.
 *   The array (FP8Q_STATS_NOALLOC_ROWS rows of 3 doubles, 96 KiB) is held
 *   by every GPU that loads the library until the process exits.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.  The address is looked up again only when
 *   the device's context has been re-created (after a cudaDeviceReset).
 *   One CTA per row of the array: 4 per SM, or one per 2^20 elements when
 *   that is more.
 *   All calls share the one array, which keeps the contents of the last
 *   call: calls that overlap on the GPU (two streams, or two host threads)
 *   race on it and give wrong results, so order them on one stream. */
#define FP8Q_STATS_NOALLOC_ROWS 4096
#define FP8Q_STATS_NOALLOC_MAX_N (4096LL << 20)
FP8Q_API int fp8q_error_stats_noalloc(const void* x, int dtype, int64_t n, const uint8_t* q,
                                      int format, const float* d_scale_inv, double* d_out,
                                      void* stream);

/* Number of pipeline waits on the current device that ran out of time since
 * the last call (and reset it).  Kernels that stage tiles through TMA
 * (column-wise mx_cast_ex, mx_cast_dual, fp8q_cast_transpose) bound every
 * wait for a tile; on timeout they count it here and stop instead of
 * hanging, leaving their outputs incomplete.  A healthy run reads 0.
 * Synchronous. */
FP8Q_API int fp8q_pipeline_status(unsigned int* timed_out_waits);

/* Diagnostic of the timeout path: two launches, each waiting on a pipeline
 * barrier that nothing completes -- a bare bounded wait, and the per-warp
 * tile pipeline of the TMA-staged kernels with no load issued.  Each wait
 * gives up (after about half a second) and is counted, so
 * fp8q_pipeline_status reports two more timed-out waits; the device stays
 * usable. */
FP8Q_API int fp8q_pipeline_selftest(void* stream);

/* Name of a status code (static string). */
FP8Q_API const char* fp8q_strerror(int code);

/* Text of the last CUDA error seen by the calling thread ("" if none). */
FP8Q_API const char* fp8q_last_cuda_error(void);

/* Number of kernels this library has launched in this process. */
FP8Q_API long long fp8q_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8Q_H */

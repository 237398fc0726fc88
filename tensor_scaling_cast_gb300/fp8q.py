"""Thin Python binding of libfp8q's C ABI (argument marshalling only).

Every function here has the name of the C entry point it calls and does no
arithmetic of the method: it turns torch tensors into device pointers, the
current torch stream into a ``cudaStream_t`` and a non-zero status into an
exception.  There is no CPU path: if ``libfp8q.so`` is missing or no GPU is
usable the calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfp8q.so")

E4M3, E5M2 = 0, 1
MX_FLOOR, MX_CEIL, MX_NEAREST = 0, 1, 2
MX_ROWWISE, MX_COLWISE = 0, 1
EST_MAX_WINDOW, EST_SMOOTHED = 0, 1
F32, BF16 = 0, 1
NO_EXP = -(2 ** 31)
MAX_WINDOW = 256

_STATUS = {0: "FP8Q_OK", -1: "FP8Q_EINVAL", -2: "FP8Q_EALIGN", -3: "FP8Q_EDTYPE", -4: "FP8Q_ECUDA",
           -5: "FP8Q_EHANDLE", -6: "FP8Q_ENOMEM", -7: "FP8Q_EDEVICE", -8: "FP8Q_ESIZE"}


class Fp8qError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        self.status = status
        msg = f"{what} failed: {_STATUS.get(status, status)}"
        super().__init__(msg + (f" ({detail})" if detail else ""))


_lib = None


def load() -> ctypes.CDLL:
    """Load libfp8q.so (built by ``__graft_entry__.build()`` or
    ``tensor_scaling_cast_gb300.build``).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run tensor_scaling_cast_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    p, i, i64, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    L.fp8q_create.argtypes = [i, i, i, i, ctypes.POINTER(p)]
    L.fp8q_create_ex.argtypes = [i, i, i, i, i, f, i, ctypes.POINTER(p)]
    L.fp8q_get_estimator_state.argtypes = [p, ctypes.POINTER(f), ctypes.POINTER(i),
                                           ctypes.POINTER(ctypes.c_longlong)]
    L.fp8q_set_estimator_state.argtypes = [p, f, i, ctypes.c_longlong]
    L.fp8q_destroy.argtypes = [p]
    L.fp8q_cast.argtypes = [p, p, i, i64, p, p, p, p, p]
    L.fp8q_cast_multi.argtypes = [p, p, p, p, p, p, p, p, i, p]
    L.fp8q_cast_multi_ex.argtypes = [p, p, p, p, p, p, p, p, p, p, i, p]
    L.fp8q_loss_scaler_create.argtypes = [f, i, f, f, ctypes.POINTER(p)]
    L.fp8q_loss_scaler_destroy.argtypes = [p]
    L.fp8q_loss_scaler_update.argtypes = [p, p, i, p, p, p]
    L.fp8q_loss_scaler_read.argtypes = [p, ctypes.POINTER(f), ctypes.POINTER(i)]
    L.mx_cast.argtypes = [p, i, i64, i64, i, i, p, p, p, p]
    L.mx_cast_ex.argtypes = [p, i, i64, i64, i, i, i, i, p, p, p, p]
    L.mx_cast_dual.argtypes = [p, i, i64, i64, i, i, i, p, p, p, p, p, p, p]
    L.fp8q_cast_transpose.argtypes = [p, p, i, i64, i64, p, p, p, p, p, p]
    L.fp8q_amax_history.argtypes = [p, ctypes.POINTER(f), i, ctypes.POINTER(i)]
    L.fp8q_scale_state.argtypes = [p, ctypes.POINTER(i), ctypes.POINTER(ctypes.c_longlong)]
    L.fp8q_set_history.argtypes = [p, ctypes.POINTER(f), i, i]
    L.fp8q_reset.argtypes = [p]
    L.fp8q_error_stats.argtypes = [p, i, i64, p, i, p, p, p]
    L.mx_error_stats.argtypes = [p, i, i64, i64, p, p, i, p, p]
    L.fp8q_error_stats_noalloc.argtypes = [p, i, i64, p, i, p, p, p]
    L.fp8q_pipeline_status.argtypes = [ctypes.POINTER(ctypes.c_uint)]
    L.fp8q_pipeline_status.restype = i
    L.fp8q_pipeline_selftest.argtypes = [p]
    L.fp8q_pipeline_selftest.restype = i
    L.fp8q_strerror.argtypes = [i]
    L.fp8q_strerror.restype = ctypes.c_char_p
    L.fp8q_last_cuda_error.restype = ctypes.c_char_p
    L.fp8q_launch_count.restype = ctypes.c_longlong
    for name in ("mx_cast_dual", "fp8q_cast_transpose", "fp8q_cast_multi_ex", "fp8q_loss_scaler_create", "fp8q_loss_scaler_destroy",
                 "fp8q_loss_scaler_update", "fp8q_loss_scaler_read",
                 "fp8q_create", "fp8q_create_ex", "fp8q_get_estimator_state",
                 "fp8q_set_estimator_state", "fp8q_destroy", "fp8q_cast", "fp8q_cast_multi", "mx_cast", "mx_cast_ex",
                 "fp8q_amax_history", "fp8q_scale_state", "fp8q_set_history", "fp8q_reset",
                 "fp8q_error_stats", "mx_error_stats", "fp8q_error_stats_noalloc"):
        getattr(L, name).restype = i
    _lib = L
    return L


def _check(status: int, what: str):
    if status != 0:
        detail = ""
        if status == -4:
            detail = load().fp8q_last_cuda_error().decode()
        raise Fp8qError(status, what, detail)


# The entry points declare their pointer arguments as c_void_p, so plain
# Python ints (and None for NULL) are passed straight through.
def _ptr(t):
    return None if t is None else t.data_ptr()


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported input dtype {t.dtype}: bf16 or fp32")


# torch's raw getter of the current stream (the public path builds a Stream
# object per call); falls back to the public path where it is absent.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(torch.cuda.current_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def fp8q_pipeline_status() -> int:
    """Pipeline waits that timed out on the current device since the last call."""
    n = ctypes.c_uint()
    _check(load().fp8q_pipeline_status(ctypes.byref(n)), "fp8q_pipeline_status")
    return n.value


def fp8q_pipeline_selftest(stream=None):
    """Launch the never-completed barrier wait (see the C header)."""
    _check(load().fp8q_pipeline_selftest(_stream(stream)), "fp8q_pipeline_selftest")


def launch_count() -> int:
    return int(load().fp8q_launch_count())


# ---- handles ---------------------------------------------------------------

def fp8q_create(fmt: int, window: int, margin: int = 0, hysteresis: int = 0) -> int:
    h = ctypes.c_void_p()
    _check(load().fp8q_create(fmt, window, margin, hysteresis, ctypes.byref(h)), "fp8q_create")
    return h.value


def fp8q_create_ex(fmt: int, window: int, margin: int = 0, hysteresis: int = 0,
                   estimator: int = EST_MAX_WINDOW, alpha: float = 1.0, interval: int = 1) -> int:
    h = ctypes.c_void_p()
    _check(load().fp8q_create_ex(fmt, window, margin, hysteresis, estimator, alpha, interval,
                                 ctypes.byref(h)), "fp8q_create_ex")
    return h.value


def fp8q_get_estimator_state(h: int):
    """(running average or None, number of casts)."""
    a, ha, st = ctypes.c_float(), ctypes.c_int(), ctypes.c_longlong()
    _check(load().fp8q_get_estimator_state(h, ctypes.byref(a), ctypes.byref(ha),
                                           ctypes.byref(st)), "fp8q_get_estimator_state")
    return (a.value if ha.value else None), st.value


def fp8q_set_estimator_state(h: int, average, steps: int):
    _check(load().fp8q_set_estimator_state(h, 0.0 if average is None else average,
                                           0 if average is None else 1, steps),
           "fp8q_set_estimator_state")


def fp8q_destroy(h: int):
    _check(load().fp8q_destroy(h), "fp8q_destroy")


def fp8q_cast(h: int, x: torch.Tensor, q: torch.Tensor, scale_inv=None, amax=None, clipped=None,
              stream=None):
    """x: contiguous bf16/fp32 CUDA tensor; q: uint8 CUDA tensor of x.numel()
    bytes; scale_inv / amax: float32 CUDA scalars; clipped: int64 CUDA scalar
    (read as uint64)."""
    _check(load().fp8q_cast(h, _ptr(x), _dtype(x), x.numel(), _ptr(q),
                            _ptr(scale_inv), _ptr(amax), _ptr(clipped), _stream(stream)),
           "fp8q_cast")


def fp8q_cast_multi(hs, xs, qs, scale_inv=None, amax=None, clipped=None, stream=None):
    """hs: handles; xs / qs: lists of CUDA tensors; scale_inv / amax: float32
    CUDA tensors [count]; clipped: int64 CUDA tensor [count]."""
    n = len(hs)
    H = (ctypes.c_void_p * n)(*hs)
    X = (ctypes.c_void_p * n)(*[x.data_ptr() for x in xs])
    Q = (ctypes.c_void_p * n)(*[q.data_ptr() for q in qs])
    D = (ctypes.c_int * n)(*[_dtype(x) for x in xs])
    N = (ctypes.c_int64 * n)(*[x.numel() for x in xs])
    _check(load().fp8q_cast_multi(H, X, D, N, Q, _ptr(scale_inv), _ptr(amax), _ptr(clipped), n,
                                  _stream(stream)), "fp8q_cast_multi")


def fp8q_cast_multi_ex(hs, xs, qs, scale_inv=None, amax=None, clipped=None, nonfinite=None,
                       underflow=None, stream=None):
    """fp8q_cast_multi plus int64 CUDA tensors [count] of non-finite and
    underflow counts (either may be None)."""
    n = len(hs)
    H = (ctypes.c_void_p * n)(*hs)
    X = (ctypes.c_void_p * n)(*[x.data_ptr() for x in xs])
    Q = (ctypes.c_void_p * n)(*[q.data_ptr() for q in qs])
    D = (ctypes.c_int * n)(*[_dtype(x) for x in xs])
    N = (ctypes.c_int64 * n)(*[x.numel() for x in xs])
    _check(load().fp8q_cast_multi_ex(H, X, D, N, Q, _ptr(scale_inv), _ptr(amax), _ptr(clipped),
                                     _ptr(nonfinite), _ptr(underflow), n, _stream(stream)),
           "fp8q_cast_multi_ex")


def fp8q_loss_scaler_create(init_scale: float, growth_interval: int, min_scale: float = 1.0,
                            max_scale: float = 2.0 ** 24) -> int:
    h = ctypes.c_void_p()
    _check(load().fp8q_loss_scaler_create(init_scale, growth_interval, min_scale, max_scale,
                                          ctypes.byref(h)), "fp8q_loss_scaler_create")
    return h.value


def fp8q_loss_scaler_destroy(h: int):
    _check(load().fp8q_loss_scaler_destroy(h), "fp8q_loss_scaler_destroy")


def fp8q_loss_scaler_update(h: int, nonfinite: torch.Tensor, scale=None, skip=None, stream=None):
    """nonfinite: int64 CUDA tensor of counts; scale: float32 CUDA scalar;
    skip: int32 CUDA scalar."""
    _check(load().fp8q_loss_scaler_update(h, _ptr(nonfinite), nonfinite.numel(),
                                          _ptr(scale), _ptr(skip), _stream(stream)),
           "fp8q_loss_scaler_update")


def fp8q_loss_scaler_read(h: int):
    """(scale, clean-step streak)."""
    sc, g = ctypes.c_float(), ctypes.c_int()
    _check(load().fp8q_loss_scaler_read(h, ctypes.byref(sc), ctypes.byref(g)),
           "fp8q_loss_scaler_read")
    return sc.value, g.value


def mx_cast(x: torch.Tensor, fmt: int, headroom: int, q: torch.Tensor, e8m0: torch.Tensor,
            clipped=None, stream=None):
    rows, cols = x.shape
    _check(load().mx_cast(_ptr(x), _dtype(x), rows, cols, fmt, headroom, _ptr(q), _ptr(e8m0),
                          _ptr(clipped), _stream(stream)), "mx_cast")


def mx_cast_ex(x: torch.Tensor, fmt: int, rule: int, headroom: int, axis: int, q: torch.Tensor,
               e8m0: torch.Tensor, clipped=None, stream=None):
    """axis MX_ROWWISE: e8m0 [rows, cols/32]; MX_COLWISE: e8m0 [rows/32, cols]."""
    rows, cols = x.shape
    _check(load().mx_cast_ex(_ptr(x), _dtype(x), rows, cols, fmt, rule, headroom, axis, _ptr(q),
                             _ptr(e8m0), _ptr(clipped), _stream(stream)), "mx_cast_ex")


def mx_cast_dual(x: torch.Tensor, fmt: int, rule: int, headroom: int, q_row, e8_row, q_colt, e8_colt,
                 clipped_row=None, clipped_col=None, stream=None):
    """Row-wise MX of x and row-wise MX of x^T (column-wise blocks written
    transposed) from one read: q_row [rows, cols], e8_row [rows, cols/32],
    q_colt [cols, rows], e8_colt [cols, rows/32]."""
    rows, cols = x.shape
    _check(load().mx_cast_dual(_ptr(x), _dtype(x), rows, cols, fmt, rule, headroom, _ptr(q_row),
                               _ptr(e8_row), _ptr(q_colt), _ptr(e8_colt), _ptr(clipped_row),
                               _ptr(clipped_col), _stream(stream)), "mx_cast_dual")


def fp8q_cast_transpose(h: int, x: torch.Tensor, q, qt, scale_inv=None, amax=None, clipped=None,
                        stream=None):
    """Per-tensor cast of x [rows, cols] to q [rows, cols] and qt [cols, rows]."""
    rows, cols = x.shape
    _check(load().fp8q_cast_transpose(h, _ptr(x), _dtype(x), rows, cols, _ptr(q),
                                      _ptr(qt), _ptr(scale_inv), _ptr(amax), _ptr(clipped),
                                      _stream(stream)), "fp8q_cast_transpose")


def fp8q_amax_history(h: int, capacity: int = MAX_WINDOW) -> list[float]:
    buf = (ctypes.c_float * max(1, capacity))()
    nv = ctypes.c_int()
    _check(load().fp8q_amax_history(h, buf, capacity, ctypes.byref(nv)),
           "fp8q_amax_history")
    return [buf[i] for i in range(nv.value)]


def fp8q_scale_state(h: int):
    """(previous exponent or None, number of casts)."""
    e = ctypes.c_int()
    st = ctypes.c_longlong()
    _check(load().fp8q_scale_state(h, ctypes.byref(e), ctypes.byref(st)),
           "fp8q_scale_state")
    return (None if e.value == NO_EXP else e.value), st.value


def fp8q_set_history(h: int, values, prev_exp=None):
    buf = (ctypes.c_float * max(1, len(values)))(*values)
    _check(load().fp8q_set_history(h, buf, len(values),
                                   NO_EXP if prev_exp is None else int(prev_exp)),
           "fp8q_set_history")


def fp8q_reset(h: int):
    _check(load().fp8q_reset(h), "fp8q_reset")


def fp8q_error_stats(x: torch.Tensor, q: torch.Tensor, fmt: int, scale_inv: torch.Tensor,
                     out: torch.Tensor, stream=None):
    _check(load().fp8q_error_stats(_ptr(x), _dtype(x), x.numel(), _ptr(q), fmt, _ptr(scale_inv),
                                   _ptr(out), _stream(stream)), "fp8q_error_stats")


def fp8q_error_stats_noalloc(x: torch.Tensor, q: torch.Tensor, fmt: int, scale_inv: torch.Tensor,
                             out: torch.Tensor, stream=None):
    """fp8q_error_stats without any device allocation (fixed library
    scratch; n <= 2^32; calls must not overlap on the GPU)."""
    _check(load().fp8q_error_stats_noalloc(_ptr(x), _dtype(x), x.numel(), _ptr(q), fmt,
                                           _ptr(scale_inv), _ptr(out), _stream(stream)),
           "fp8q_error_stats_noalloc")


def mx_error_stats(x: torch.Tensor, q: torch.Tensor, e8m0: torch.Tensor, fmt: int,
                   out: torch.Tensor, stream=None):
    rows, cols = x.shape
    _check(load().mx_error_stats(_ptr(x), _dtype(x), rows, cols, _ptr(q), _ptr(e8m0), fmt,
                                 _ptr(out), _stream(stream)), "mx_error_stats")


# ---- convenience wrapper ---------------------------------------------------

class ScaledCast:
    """One tensor's scaling state on the GPU (owns an fp8q handle) with
    output buffers allocated by torch."""

    def __init__(self, fmt: int, window: int, margin: int = 0, hysteresis: int = 0,
                 estimator: int = EST_MAX_WINDOW, alpha: float = 1.0, interval: int = 1):
        self.fmt, self.window, self.margin, self.hysteresis = fmt, window, margin, hysteresis
        self.handle = fp8q_create_ex(fmt, window, margin, hysteresis, estimator, alpha, interval)

    def __call__(self, x: torch.Tensor, q: torch.Tensor | None = None, stream=None):
        """Returns (q uint8, scale_inv f32[1], amax f32[1], clipped i64[1]) on x's device."""
        dev = x.device
        if q is None:
            q = torch.empty(x.shape, dtype=torch.uint8, device=dev)
        # one 16-byte allocation: scale_inv f32, amax f32, clipped i64
        outs = torch.empty(4, dtype=torch.float32, device=dev)
        scale_inv, amax, clipped = outs[0:1], outs[1:2], outs[2:4].view(torch.int64)
        fp8q_cast(self.handle, x, q, scale_inv, amax, clipped, stream)
        return q, scale_inv, amax, clipped

    def history(self):
        return fp8q_amax_history(self.handle, max(1, self.window))

    def state(self):
        return fp8q_scale_state(self.handle)

    def set_history(self, values, prev_exp=None):
        fp8q_set_history(self.handle, values, prev_exp)

    def reset(self):
        fp8q_reset(self.handle)

    def close(self):
        if self.handle:
            fp8q_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

"""ctypes binding of the plain-C oracle (``oracle/oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg; never by the product library.  Arrays are numpy
arrays of raw bit patterns: fp32 inputs as uint32, bf16 inputs as uint16.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "oracle.c")
LIB = os.path.join(_HERE, "_build", "liboracle.so")

F32, BF16 = 0, 1
E4M3, E5M2, FP16 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile oracle.c with the host C compiler (gcc, OpenMP)."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                           "-o", tmp, SRC, "-lm"])
    os.replace(tmp, LIB)
    return LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB)
        c_i64, c_u32, c_int, c_p = ctypes.c_int64, ctypes.c_uint32, ctypes.c_int, ctypes.c_void_p
        L.orc_decode.argtypes = [c_int, c_u32]
        L.orc_decode.restype = ctypes.c_double
        L.orc_encode_double.argtypes = [c_int, ctypes.c_double, ctypes.POINTER(c_int)]
        L.orc_encode_double.restype = c_u32
        L.orc_cast_scalar.argtypes = [c_int, c_u32, c_int, ctypes.POINTER(c_int)]
        L.orc_cast_scalar.restype = c_u32
        L.orc_amax.argtypes = [c_p, c_int, c_i64, c_int]
        L.orc_amax.restype = c_u32
        L.orc_cast.argtypes = [c_p, c_int, c_i64, c_int, c_int, c_p, ctypes.POINTER(c_u32), c_int]
        L.orc_cast.restype = c_i64
        L.orc_cast_at.argtypes = [c_p, c_int, c_p, c_i64, c_int, c_int, c_p, c_p]
        L.orc_cast_at.restype = None
        L.orc_scale_exp.argtypes = [c_u32, c_int, c_int, ctypes.POINTER(c_int)]
        L.orc_scale_exp.restype = c_int
        L.orc_mx_exp.argtypes = [c_u32, c_int, c_int]
        L.orc_mx_exp.restype = c_int
        L.orc_mx_cast.argtypes = [c_p, c_int, c_i64, c_i64, c_int, c_int, c_p, c_p, c_int]
        L.orc_mx_cast.restype = c_i64
        L.orc_mx_exp_rule.argtypes = [c_u32, c_int, c_int, c_int]
        L.orc_mx_exp_rule.restype = c_int
        L.orc_mx_cast_ex.argtypes = [c_p, c_int, c_i64, c_i64, c_int, c_int, c_int, c_int, c_p, c_p, c_int]
        L.orc_mx_cast_ex.restype = c_i64
        L.orc_count_special.argtypes = [c_p, c_int, c_i64, c_p, ctypes.POINTER(c_i64), ctypes.POINTER(c_i64)]
        L.orc_count_special.restype = None
        L.orc_stats.argtypes = [c_p, c_int, c_i64, c_p, c_int, c_int, c_p, c_int]
        L.orc_stats.restype = None
        L.orc_mx_stats.argtypes = [c_p, c_int, c_i64, c_i64, c_p, c_p, c_int, c_p, c_int]
        L.orc_mx_stats.restype = None
        _lib = L
    return _lib


def _dtype_of(x: np.ndarray) -> int:
    if x.dtype == np.uint32:
        return F32
    if x.dtype == np.uint16:
        return BF16
    raise TypeError("oracle inputs are raw bits: uint32 (fp32) or uint16 (bf16)")


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def decode(fmt: int, code: int) -> float:
    return lib().orc_decode(fmt, code)


def encode_double(fmt: int, v: float):
    c = ctypes.c_int()
    code = lib().orc_encode_double(fmt, float(v), ctypes.byref(c))
    return int(code), bool(c.value)


def cast_scalar(fmt: int, xbits: int, e: int):
    c = ctypes.c_int()
    code = lib().orc_cast_scalar(fmt, xbits, e, ctypes.byref(c))
    return int(code), bool(c.value)


def amax(x: np.ndarray, nthreads: int = 1) -> int:
    x = np.ascontiguousarray(x)
    return int(lib().orc_amax(_ptr(x), _dtype_of(x), x.size, nthreads))


def cast(x: np.ndarray, fmt: int, e: int, nthreads: int = 1):
    """Returns (q uint8[n], amax_bits, clipped)."""
    x = np.ascontiguousarray(x)
    q = np.empty(x.size, dtype=np.uint8)
    a = ctypes.c_uint32()
    clipped = lib().orc_cast(_ptr(x), _dtype_of(x), x.size, fmt, e, _ptr(q), ctypes.byref(a), nthreads)
    return q.reshape(x.shape), int(a.value), int(clipped)


def cast_at(x: np.ndarray, idx: np.ndarray, fmt: int, e: int):
    """Cast only x.flat[idx]; returns (q uint8[m], clip uint8[m])."""
    x = np.ascontiguousarray(x)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    q = np.empty(idx.size, dtype=np.uint8)
    cl = np.empty(idx.size, dtype=np.uint8)
    lib().orc_cast_at(_ptr(x), _dtype_of(x), _ptr(idx), idx.size, fmt, e, _ptr(q), _ptr(cl))
    return q, cl


def scale_exp(amax_bits: int, fmt: int, margin: int):
    """Exponent from the definition, or None for a zero / non-finite amax."""
    ok = ctypes.c_int()
    e = lib().orc_scale_exp(amax_bits, fmt, margin, ctypes.byref(ok))
    return int(e) if ok.value else None


def mx_exp(amax_bits: int, fmt: int, headroom: int) -> int:
    return int(lib().orc_mx_exp(amax_bits, fmt, headroom))


def mx_cast(x: np.ndarray, fmt: int, headroom: int, nthreads: int = 1):
    """x: [rows, cols] raw bits.  Returns (q [rows, cols], e8m0 [rows, cols/32], clipped)."""
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    q = np.empty((rows, cols), dtype=np.uint8)
    e8 = np.empty((rows, cols // 32), dtype=np.uint8)
    clipped = lib().orc_mx_cast(_ptr(x), _dtype_of(x), rows, cols, fmt, headroom, _ptr(q), _ptr(e8), nthreads)
    return q, e8, int(clipped)


def stats(x: np.ndarray, q: np.ndarray, fmt: int, e: int, nthreads: int = 1):
    """(mse, bias, finite count) of decode(q) * 2^-e against x."""
    x = np.ascontiguousarray(x)
    q = np.ascontiguousarray(q)
    out = np.zeros(3, dtype=np.float64)
    lib().orc_stats(_ptr(x), _dtype_of(x), x.size, _ptr(q), fmt, e, _ptr(out), nthreads)
    return float(out[0]), float(out[1]), int(out[2])


def mx_stats(x: np.ndarray, q: np.ndarray, e8: np.ndarray, fmt: int, nthreads: int = 1):
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    out = np.zeros(3, dtype=np.float64)
    lib().orc_mx_stats(_ptr(x), _dtype_of(x), rows, cols, _ptr(np.ascontiguousarray(q)),
                       _ptr(np.ascontiguousarray(e8)), fmt, _ptr(out), nthreads)
    return float(out[0]), float(out[1]), int(out[2])


MX_FLOOR, MX_CEIL, MX_NEAREST = 0, 1, 2
ROWWISE, COLWISE = 0, 1


def mx_exp_rule(amax_bits: int, fmt: int, rule: int, headroom: int) -> int:
    return int(lib().orc_mx_exp_rule(amax_bits, fmt, rule, headroom))


def mx_cast_ex(x: np.ndarray, fmt: int, rule: int, headroom: int, axis: int, nthreads: int = 1):
    """x: [rows, cols] raw bits.  axis 0: e8m0 [rows, cols/32]; axis 1:
    e8m0 [rows/32, cols].  Returns (q [rows, cols], e8m0, clipped)."""
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    q = np.empty((rows, cols), dtype=np.uint8)
    e8 = np.empty((rows, cols // 32) if axis == 0 else (rows // 32, cols), dtype=np.uint8)
    clipped = lib().orc_mx_cast_ex(_ptr(x), _dtype_of(x), rows, cols, fmt, rule, headroom, axis,
                                   _ptr(q), _ptr(e8), nthreads)
    return q, e8, int(clipped)


def count_special(x: np.ndarray, q: np.ndarray):
    """(non-finite inputs, underflowed elements) of a cast x -> q."""
    x = np.ascontiguousarray(x).reshape(-1)
    q = np.ascontiguousarray(q).reshape(-1)
    nf, uf = ctypes.c_int64(), ctypes.c_int64()
    lib().orc_count_special(_ptr(x), _dtype_of(x), x.size, _ptr(q), ctypes.byref(nf), ctypes.byref(uf))
    return int(nf.value), int(uf.value)


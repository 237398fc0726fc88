"""The C-ABI library builds for sm_103a, loads, and exports every entry point
that include/fp8q.h declares; host-side argument checks answer without a GPU."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8q.h")


def declared_symbols():
    src = open(HEADER).read()
    return re.findall(r"FP8Q_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)


@pytest.fixture(scope="module")
def lib():
    from tensor_scaling_cast_gb300 import build
    build.build()
    from tensor_scaling_cast_gb300 import fp8q
    return fp8q.load()


def test_header_declares_the_api():
    names = set(declared_symbols())
    for n in ("fp8q_create", "fp8q_destroy", "fp8q_cast", "fp8q_cast_multi", "mx_cast",
              "fp8q_amax_history", "fp8q_set_history", "fp8q_error_stats", "mx_error_stats"):
        assert n in names


def test_exports_every_declared_symbol(lib):
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert missing == []


def test_built_for_sm_103a():
    from tensor_scaling_cast_gb300 import build
    assert "arch=compute_103a,code=sm_103a" in build.ARCH


def test_host_argument_checks(lib):
    """Checks that run before any CUDA call."""
    h = ctypes.c_void_p()
    assert lib.fp8q_create(7, 16, 0, 0, ctypes.byref(h)) == -3          # bad format
    assert lib.fp8q_create(0, 257, 0, 0, ctypes.byref(h)) == -1         # window too large
    assert lib.fp8q_create(0, -1, 0, 0, ctypes.byref(h)) == -1
    assert lib.fp8q_create(0, 4, -1, 0, ctypes.byref(h)) == -1
    assert lib.fp8q_create(0, 4, 0, 0, None) == -1
    assert lib.mx_cast(None, 1, 4, 48, 0, 0, None, None, None, None) == -1   # cols % 32
    assert lib.mx_cast(None, 1, 4, 64, 0, 9, None, None, None, None) == -1   # headroom
    assert lib.mx_cast(None, 5, 4, 64, 0, 0, None, None, None, None) == -3   # dtype
    assert lib.mx_cast(ctypes.c_void_p(0x1008), 1, 1, 32, 0, 0, ctypes.c_void_p(0x2000),
                       ctypes.c_void_p(0x3000), None, None) == -2             # misaligned x
    assert lib.fp8q_cast(None, None, 1, 0, None, None, None, None, None) == -5  # null handle
    assert lib.fp8q_cast_multi(None, None, None, None, None, None, None, None, 0, None) == -1
    assert lib.fp8q_destroy(None) == 0
    assert lib.fp8q_strerror(-2) == b"pointer not 16-byte aligned"


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU answer")
def test_no_gpu_means_an_error_not_a_fallback(lib):
    h = ctypes.c_void_p()
    assert lib.fp8q_create(0, 16, 0, 0, ctypes.byref(h)) == -4          # FP8Q_ECUDA
    assert h.value is None
    assert lib.fp8q_last_cuda_error() != b""

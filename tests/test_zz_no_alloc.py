"""The allocation-free statistics entry point, fp8q_error_stats_noalloc.

Some callers of this library cannot allocate device memory at the moment they
want error statistics: their own caching allocator owns the device's memory,
they run right after an out-of-memory error, or an allocation would stall a
latency-bound loop.  fp8q_error_stats takes its per-CTA partial sums from
cudaMallocAsync; the no-alloc variant takes them from a fixed array inside
the library.  This file checks, through the C ABI, that the variant gives
the same statistics as fp8q_error_stats (within the 1e-6 relative tolerance
the other statistics tests use) on two different calls in a row -- the
second smaller than the first, so rows left over from the first call must
not leak into it -- and that it rejects a size beyond its limit.

Named to be collected last: a run that stops at the first failure has run
every other test before this one.
"""
import ctypes

import pytest
import torch

from tensor_scaling_cast_gb300 import fp8q as F
from tensor_scaling_cast_gb300 import synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the gpu tests")
    from tensor_scaling_cast_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    return F.load()


def _cast(x, fmt):
    g = F.ScaledCast(fmt, window=1)
    g(x * 0.125)                                   # small window amax: the next cast clips
    q, sinv, _, _ = g(x)
    g.close()
    return q, sinv


def _close(a, b):
    mse, bias, n = a
    mse_r, bias_r, n_r = b
    return (n == n_r and abs(mse - mse_r) <= 1e-6 * mse_r
            and abs(bias - bias_r) <= 1e-6 * max(abs(bias_r), mse_r ** 0.5))


def _noalloc(lib, x, q, fmt, sinv, out):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dt = 1 if x.dtype == torch.bfloat16 else 0
    return lib.fp8q_error_stats_noalloc(ctypes.c_void_p(x.data_ptr()), dt, x.numel(),
                                        ctypes.c_void_p(q.data_ptr()), fmt,
                                        ctypes.c_void_p(sinv.data_ptr()),
                                        ctypes.c_void_p(out.data_ptr()), stream)


def test_noalloc_stats_match_allocating_entry_point(lib):
    cases = [
        (synthetic.spike_step(9, "cuda", shape=(4096, 2048)), 0),    # 8 Mi elements: 8 rows
        (synthetic.spike_step(3, "cuda", shape=(1000, 1000)).float(), 1),  # 1e6: 1 row
    ]
    for x, fmt in cases:                           # two calls in a row
        q, sinv = _cast(x, fmt)
        ref = torch.empty(3, dtype=torch.float64, device="cuda")
        F.fp8q_error_stats(x, q, fmt, sinv, ref)
        out = torch.full((3,), float("nan"), dtype=torch.float64, device="cuda")
        assert _noalloc(lib, x, q, fmt, sinv, out) == 0
        torch.cuda.synchronize()
        assert _close(out.cpu().tolist(), ref.cpu().tolist()), (out, ref)


def test_noalloc_stats_rejects_size_above_limit(lib):
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(16, dtype=torch.uint8, device="cuda")
    s = torch.ones(1, dtype=torch.float32, device="cuda")
    out = torch.zeros(3, dtype=torch.float64, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # the size check comes before any device access: n is only compared
    st = lib.fp8q_error_stats_noalloc(ctypes.c_void_p(x.data_ptr()), 1, (4096 << 20) + 1,
                                      ctypes.c_void_p(q.data_ptr()), 0,
                                      ctypes.c_void_p(s.data_ptr()),
                                      ctypes.c_void_p(out.data_ptr()), stream)
    assert st == -8
    assert lib.fp8q_strerror(-8) == b"size above the fixed scratch limit"

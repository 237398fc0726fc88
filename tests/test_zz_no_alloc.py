"""The allocation-free statistics entry point, fp8q_error_stats_noalloc.

Some callers of this library cannot allocate device memory at the moment they
want error statistics: their own caching allocator owns the device's memory,
they run right after an out-of-memory error, or an allocation would stall a
latency-bound loop.  fp8q_error_stats takes its per-CTA partial sums from
cudaMallocAsync; the no-alloc variant takes them from a fixed array inside
the library.  This file checks, through the C ABI, that the variant gives
the statistics of the CPU oracle and of fp8q_error_stats -- MSE and bias
within 1e-6 relative, the count exact -- on calls made in a row, each
smaller than the one before, so partial sums left in the array by an
earlier call must not leak into a later one; and that it rejects a size
beyond its limit.

Named to be collected last: a run that stops at the first failure has run
every other test before this one.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

from canary import Guards
from oracle import coracle
from tensor_scaling_cast_gb300 import fp8q as F
from tensor_scaling_cast_gb300 import synthetic

pytestmark = pytest.mark.gpu

NT = os.cpu_count() or 1
G = Guards(seed=0x20)


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the gpu tests")
    from tensor_scaling_cast_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    return F.load()


def _cast(x, fmt):
    """A clipping per-tensor cast: the window holds a smaller tensor's amax."""
    g = F.ScaledCast(fmt, window=1)
    g(x * 0.125)
    q, sinv, _, clipped = g(x)
    torch.cuda.synchronize()
    assert int(clipped.item()) > 0
    g.close()
    return q, sinv


def _rel_close(a, b):
    """Every statistic within 1e-6 relative of the reference (an exact zero
    must be met exactly) and the counts equal."""
    (mse, bias, n), (mse_r, bias_r, n_r) = a, b
    return (int(n) == int(n_r) and abs(mse - mse_r) <= 1e-6 * abs(mse_r)
            and abs(bias - bias_r) <= 1e-6 * abs(bias_r))


def _noalloc(lib, x, q, fmt, sinv, out):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dt = 1 if x.dtype == torch.bfloat16 else 0
    return lib.fp8q_error_stats_noalloc(ctypes.c_void_p(x.data_ptr()), dt, x.numel(),
                                        ctypes.c_void_p(q.data_ptr()), fmt,
                                        ctypes.c_void_p(sinv.data_ptr()),
                                        ctypes.c_void_p(out.data_ptr()), stream)


def _host_bits(x):
    x = x.detach().contiguous().cpu()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    return x.view(torch.int32).numpy().view(np.uint32).reshape(-1)


def test_noalloc_stats_match_oracle_and_allocating_entry_point(lib):
    cases = [
        # 640 Mi + 12,345 bf16 elements: 641 slabs of 2^20, more CTAs than 4 per SM
        (synthetic.mx_tanh("cuda", shape=((640 << 20) + 12345,), seed=4100), 0),
        (synthetic.spike_step(9, "cuda", shape=(4096, 2048)), 1),          # 8 Mi: 4 CTAs per SM
        (synthetic.spike_step(3, "cuda", shape=(1000, 1000)).float(), 0),  # fp32, 1e6 elements
    ]
    for x, fmt in cases:                           # calls in a row, each smaller
        q, sinv = _cast(x, fmt)
        ref = torch.empty(3, dtype=torch.float64, device="cuda")
        F.fp8q_error_stats(x, q, fmt, sinv, ref)
        out = G.full(3, float("nan"), torch.float64)
        assert _noalloc(lib, x, q, fmt, sinv, out) == 0
        G.check("after fp8q_error_stats_noalloc")
        got = out.cpu().tolist()
        e = -int(np.log2(sinv.item()))
        want = coracle.stats(_host_bits(x), q.cpu().numpy().reshape(-1), fmt, e, NT)
        assert _rel_close(got, want), (x.numel(), got, want)
        assert _rel_close(got, ref.cpu().tolist()), (x.numel(), got, ref)
        G.release()
        del x, q, ref
        torch.cuda.empty_cache()


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

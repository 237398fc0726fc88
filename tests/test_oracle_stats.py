"""Dequantised-error statistics of the oracle ("what actually breaks low
precision training", "What the measurements said": error size and bias
measured separately) against exact rational arithmetic."""
from fractions import Fraction

import numpy as np

from oracle import spec


def _bf16(x):
    b = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    return ((b + ((b >> 16) & 1) + 0x7FFF) >> 16).astype(np.uint16)


def test_per_tensor_stats_exact(orc):
    rng = np.random.default_rng(31)
    x = _bf16(rng.standard_normal(3000) * 3)
    x[7] = 0x7FC0                                  # NaN input: skipped
    for f, sf in ((0, spec.E4M3), (1, spec.E5M2)):
        for e in (3, 6, 9):                        # e = 9 clips some elements
            q, _, _ = orc.cast(x, f, e)
            mse, bias, n = orc.stats(x, q, f, e)
            vals = [spec.bf16_bits_exact(int(b)) for b in x]
            mse_s, bias_s, n_s = spec.error_stats(sf, vals, list(q), lambda i: Fraction(2) ** -e)
            assert n == n_s == 2999
            assert abs(mse - float(mse_s)) <= 1e-12 * float(mse_s)
            assert abs(bias - float(bias_s)) <= 1e-12 * max(abs(float(bias_s)), float(mse_s) ** 0.5)


def test_mx_stats_exact(orc):
    rng = np.random.default_rng(32)
    x = _bf16(np.tanh(rng.standard_normal((8, 96)) * 2))
    x[2, 40] = 0x7F80                              # Inf: its block is skipped
    vals = [spec.bf16_bits_exact(int(b)) for b in x.reshape(-1)]
    for f, sf in ((0, spec.E4M3), (1, spec.E5M2)):
        for h in (0, 1):
            q, e8, _ = orc.mx_cast(x, f, h)
            mse, bias, n = orc.mx_stats(x, q, e8, f)
            e8f = e8.reshape(-1)
            scale = lambda i: None if e8f[i // 32] == 0xFF else Fraction(2) ** (int(e8f[i // 32]) - 127)
            mse_s, bias_s, n_s = spec.error_stats(sf, vals, list(q.reshape(-1)), scale)
            assert n == n_s == 8 * 96 - 32
            assert abs(mse - float(mse_s)) <= 1e-12 * float(mse_s)
            assert abs(bias - float(bias_s)) <= 1e-12 * max(abs(float(bias_s)), float(mse_s) ** 0.5)


def test_stats_zero_for_exact_values(orc):
    """Values already on the grid dequantise exactly: zero error, zero bias."""
    codes = np.array([c for c in range(256) if (c & 0x7F) < 0x7E and c != 0x80], dtype=np.uint8)
    v = np.array([orc.decode(0, int(c)) for c in codes], dtype=np.float32) * 2.0 ** -4
    x = v.astype(np.float32).view(np.uint32)
    q, _, clipped = orc.cast(x, 0, 4)
    assert clipped == 0 and np.array_equal(q, codes)
    mse, bias, n = orc.stats(x, q, 0, 4)
    assert mse == 0.0 and bias == 0.0 and n == len(codes)

"""Pins of the oracle's non-finite / underflow counts and of the dynamic
loss-scale state machine ("Mixed Precision FP16/BF16/FP8" mind-map card:
halve S and skip the step on Inf/NaN, double it after a clean streak;
"what actually breaks low precision training": underflow rates)."""
import os

import numpy as np
import pytest
import torch

from oracle import policy

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _traces():
    rows = []
    with open(os.path.join(GOLDEN, "loss_scale_traces.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                name, s0, n, flags, scales, skips = [p.strip() for p in line.split("|")]
                rows.append((name, float(s0), int(n), [int(v) for v in flags.split()],
                             [float(v) for v in scales.split()], [int(v) for v in skips.split()]))
    return rows


@pytest.mark.parametrize("row", _traces(), ids=lambda r: r[0])
def test_loss_scale_traces(row):
    name, s0, n, flags, scales, skips = row
    ls = policy.LossScaler(s0, n)
    for t, f in enumerate(flags):
        skip = ls.update([0, f, 0])
        assert (float(ls.scale), int(skip)) == (scales[t], skips[t]), (name, t)


@pytest.mark.parametrize("fmt,tdt", [(0, torch.float8_e4m3fn), (1, torch.float8_e5m2)])
def test_counts_against_library_decode(fmt, tdt, orc):
    """Underflow = finite nonzero input whose 8-bit value decodes (torch's
    float8 decode, a library routine) to zero; non-finite = NaN or Inf."""
    rng = np.random.default_rng(51)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-25, 5, 20000))).astype(np.float32)
    x[:50] = np.nan
    x[50:80] = np.inf
    x[80:90] = -np.inf
    x[90:200] = 0.0
    x[200:210] = -0.0
    for e in (0, 4, 9):
        q, _, _ = orc.cast(x.view(np.uint32), fmt, e)
        nf, uf = orc.count_special(x.view(np.uint32), q)
        dec = torch.from_numpy(q.copy()).view(tdt).to(torch.float64).numpy()
        fin = np.isfinite(x)
        assert nf == int((~fin).sum()) == 90
        assert uf == int((fin & (x != 0) & (dec == 0)).sum())
        assert uf > 0


def test_underflow_threshold_is_half_the_smallest_subnormal(orc):
    """E4M3's smallest subnormal is 2^-9: |v| <= 2^-10 rounds to zero (the
    tie goes to the even zero), anything larger does not."""
    tiny = np.array([2.0 ** -10, np.nextafter(np.float32(2.0 ** -10), np.float32(1)), -2.0 ** -10],
                    dtype=np.float32)
    q, _, _ = orc.cast(tiny.view(np.uint32), 0, 0)
    assert list(q) == [0x00, 0x01, 0x80]
    assert orc.count_special(tiny.view(np.uint32), q) == (0, 2)

"""Pins of the oracle's scaling policy ("Practice c06/E3, worked solution":
largest power of two keeping the window maximum below the format maximum
with a margin; hysteresis; the max-window of the "Max-Window Scale Estimation
..." summary)."""
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

from oracle import policy, spec

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FMAX = {0: 448.0, 1: 57344.0}


def _all_positive_finite_bf16():
    b = np.arange(1, 0x7F80, dtype=np.uint32) << 16
    return [int(x) for x in b]


@pytest.mark.parametrize("f", [0, 1])
@pytest.mark.parametrize("margin", [0, 1, 3])
def test_scale_exp_all_bf16_amax(f, margin, orc):
    """For every positive finite bf16 amax A: the C oracle's exponent equals
    floor(log2(fmax * 2^-m / A)) computed with math.frexp in exact rationals
    (clamped to [-126, 126]), and the exact spec agrees on a stride."""
    fmax = Fraction(FMAX[f])
    limit = fmax / 2 ** margin
    for i, ab in enumerate(_all_positive_finite_bf16()):
        a = spec.f32_bits_exact(ab)[1]
        e_c = orc.scale_exp(ab, f, margin)
        # closed form: ratio = limit / A; floor(log2 ratio) via frexp on the
        # exact rational (numerator and denominator are integers)
        r = limit / a
        k = r.numerator.bit_length() - r.denominator.bit_length()
        if Fraction(2) ** k > r:
            k -= 1
        elif Fraction(2) ** (k + 1) <= r:
            k += 1
        assert Fraction(2) ** k <= r < Fraction(2) ** (k + 1)
        want = max(-126, min(126, k))
        assert e_c == want, (hex(ab), e_c, want)
        if i % 97 == 0:
            assert spec.scale_exp([spec.E4M3, spec.E5M2][f], a, margin) == want


@pytest.mark.parametrize("f", [0, 1])
def test_power_of_two_leaves_at_most_factor_two(f, orc):
    """"A scale that is a power of two leaves up to a factor of two of the
    range unused" (worked solution): for any amax whose exponent is not
    clamped, fmax/2^(m+1) < 2^e * A <= fmax/2^m."""
    rng = np.random.default_rng(3)
    for margin in (0, 1, 2):
        for v in np.exp(rng.uniform(np.log(1e-30), np.log(1e30), size=4000)):
            ab = struct.unpack("<I", struct.pack("<f", v))[0]
            a = spec.f32_bits_exact(ab)[1]
            e = orc.scale_exp(ab, f, margin)
            if -126 < e < 126:
                scaled = a * Fraction(2) ** e
                assert Fraction(FMAX[f]) / 2 ** (margin + 1) < scaled <= Fraction(FMAX[f]) / 2 ** margin


def test_scale_exp_zero_and_nonfinite(orc):
    assert orc.scale_exp(0, 0, 0) is None
    assert orc.scale_exp(0x7F800000, 0, 0) is None
    assert orc.scale_exp(0x7FC00000, 1, 0) is None


def _parse_amax(s: str) -> float:
    if s == "nan":
        return float("nan")
    if "*" in s:
        a, b = s.split("*")
        return float(a) * 2.0 ** int(b.split("^")[1])
    if s.startswith("2^"):
        return 2.0 ** int(s[2:])
    return float(s)


def _traces():
    rows = []
    with open(os.path.join(GOLDEN, "window_traces.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            head, am, es, cl = [p.strip() for p in line.split("|")]
            name, fmt, w, m, h = head.split()
            rows.append((name, {"e4m3": 0, "e5m2": 1}[fmt], int(w), int(m), int(h),
                         [_parse_amax(a) for a in am.split()], [int(e) for e in es.split()],
                         None if cl == "-" else [int(c) for c in cl.split()]))
    return rows


def _step_tensor(a: float) -> np.ndarray:
    v = np.array([a, -a / 2, a / 4, -a / 8, 0.0], dtype=np.float64)
    return v.astype(np.float32).view(np.uint32)


@pytest.mark.parametrize("row", _traces(), ids=lambda r: r[0])
def test_window_traces(row):
    name, f, w, m, h, amaxes, es, clipped = row
    st = policy.ScalingState(f, w, m, h)
    for t, a in enumerate(amaxes):
        q, a_bits, sinv_bits, n_clip, e = st.step(_step_tensor(a))
        assert e == es[t], (name, t, e, es[t])
        assert policy.f32_of_bits(sinv_bits) == 2.0 ** -e
        if math.isnan(a):
            assert a_bits == 0x7FC00000
        else:
            assert policy.f32_of_bits(a_bits) == np.float32(a)
        if clipped is not None:
            assert n_clip == clipped[t], (name, t)


def test_current_scaling_never_clips(orc):
    """Current scaling picks the scale from the tensor itself, so the rule
    keeps every element in range: zero clipped for any finite tensor."""
    rng = np.random.default_rng(11)
    for trial in range(60):
        n = int(rng.integers(1, 3000))
        scale = float(np.exp(rng.uniform(-40, 40)))
        x = (rng.standard_normal(n) * scale).astype(np.float32)
        for f in (0, 1):
            st = policy.ScalingState(f, window=0, margin=int(rng.integers(0, 3)))
            _, _, _, n_clip, _ = st.step(x.view(np.uint32))
            assert n_clip == 0


def test_max_window_never_clips_below_window_max(orc):
    """Max-window guarantee (summary, "Key contributions"): when the current
    tensor's amax does not exceed the window maximum, nothing clips."""
    rng = np.random.default_rng(12)
    for f in (0, 1):
        st = policy.ScalingState(f, window=8, margin=0)
        for t in range(40):
            x = (rng.standard_normal(2000) * np.exp(rng.uniform(-3, 3))).astype(np.float32)
            cur = float(np.max(np.abs(x)))
            wmax = max(policy.f32_of_bits(b) for b in st.hist) if st.hist else None
            _, _, _, n_clip, _ = st.step(x.view(np.uint32))
            if wmax is not None and cur <= wmax:
                assert n_clip == 0


def test_spike_overflows_one_window_late(orc):
    """Most-recent scaling answers a spike one step late and the spike
    clips; a max-window that holds a larger earlier value does not clip
    ("a scale that answers a spike one window late lets the spike
    overflow")."""
    rng = np.random.default_rng(13)
    base = rng.standard_normal(4096).astype(np.float32)
    spike = base.copy()
    spike[:4] *= 8
    recent = policy.ScalingState(0, window=1)
    window = policy.ScalingState(0, window=4)
    big = base * 16
    seq = [big, base, base, spike]
    clips_recent = [recent.step(x.view(np.uint32))[3] for x in seq]
    clips_window = [window.step(x.view(np.uint32))[3] for x in seq]
    assert clips_recent[-1] > 0 and clips_window[-1] == 0


def _estimator_traces():
    rows = []
    with open(os.path.join(GOLDEN, "estimator_traces.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            head, am, es, cl = [p.strip() for p in line.split("|")]
            name, w, est, alpha, interval = head.split()
            rows.append((name, int(w), {"max": policy.MAX_WINDOW, "ema": policy.EMA}[est],
                         float(alpha), int(interval), [_parse_amax(a) for a in am.split()],
                         [int(e) for e in es.split()], [int(c) for c in cl.split()]))
    return rows


@pytest.mark.parametrize("row", _estimator_traces(), ids=lambda r: r[0])
def test_estimator_traces(row):
    name, w, est, alpha, interval, amaxes, es, clipped = row
    st = policy.ScalingState(0, w, 0, 0, estimator=est, alpha=alpha, interval=interval)
    for t, a in enumerate(amaxes):
        _, _, _, n_clip, e = st.step(_step_tensor(a))
        assert (e, n_clip) == (es[t], clipped[t]), (name, t)


def test_smoothing_with_alpha_one_is_most_recent():
    """A running average with coefficient 1 is the previous step's amax."""
    rng = np.random.default_rng(14)
    a = policy.ScalingState(0, window=0, estimator=policy.EMA, alpha=1.0)
    b = policy.ScalingState(0, window=1)
    for t in range(30):
        x = (rng.standard_normal(500) * np.exp(rng.uniform(-4, 4))).astype(np.float32).view(np.uint32)
        assert a.step(x)[4] == b.step(x)[4]


def test_interval_one_is_the_plain_policy():
    rng = np.random.default_rng(15)
    a = policy.ScalingState(1, window=4, margin=1, interval=1)
    b = policy.ScalingState(1, window=4, margin=1)
    for t in range(30):
        x = (rng.standard_normal(500) * np.exp(rng.uniform(-4, 4))).astype(np.float32).view(np.uint32)
        ra, rb = a.step(x), b.step(x)
        assert ra[3:] == rb[3:] and np.array_equal(ra[0], rb[0])


def test_smoothing_update_is_fp32_without_fma():
    """The running average is three fp32 roundings: sub, mul, add."""
    st = policy.ScalingState(0, window=0, estimator=policy.EMA, alpha=0.1)
    vals = [1.0, 3.3, 1e-3, 7.77]
    for v in vals:
        st.step(np.array([v], dtype=np.float32).view(np.uint32))
    avg = np.float32(1.0)
    for v in vals[1:]:
        d = np.float32(np.float32(v) - avg)
        avg = np.float32(avg + np.float32(np.float32(0.1) * d))
    assert st.avg == avg and st.avg.dtype == np.float32

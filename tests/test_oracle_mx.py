"""Pins of the oracle's MX cast ("what actually breaks low precision
training", "What the measurements said": blocks of 32 share a power of two
from the OCP formula, which puts the block's largest value where the 8-bit
format cannot fully reach it, so the biggest values clip; one extra bit of
exponent headroom fixes it)."""
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import spec

EMAX = {0: 8, 1: 15}


@pytest.mark.parametrize("f", [0, 1])
@pytest.mark.parametrize("h", [0, 1])
def test_mx_exp_all_bf16_amax_vs_frexp(f, h, orc):
    """E = floor(log2 A) - emax_elem + h for every positive finite bf16 A,
    floor(log2) taken from math.frexp (exact), clamped to [-127, 127]."""
    for b in range(1, 0x7F80):
        a = spec.f32_bits_exact(b << 16)[1]
        m, p = math.frexp(float(a))
        want = max(-127, min(127, (p - 1) - EMAX[f] + h))
        assert orc.mx_exp(b << 16, f, h) == want
        if b % 61 == 0:
            assert spec.mx_exp([spec.E4M3, spec.E5M2][f], a, h) == want
    assert orc.mx_exp(0, f, h) == -127


def _bf16(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bits, round to nearest even (plain integer arithmetic)."""
    b = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    r = ((b >> 16) & 1) + 0x7FFF
    return ((b + r) >> 16).astype(np.uint16)


@pytest.mark.parametrize("f", [0, 1])
def test_ocp_rule_puts_block_max_in_top_binade(f, orc):
    """Under the OCP rule the scaled block maximum lies in
    [2^emax, 2^(emax+1)): above fmax = 1.75 * 2^emax for part of that range,
    which is why the biggest values clip."""
    rng = np.random.default_rng(21)
    x = _bf16(rng.standard_normal((64, 256)) * np.exp(rng.uniform(-20, 20, size=(64, 1))))
    q, e8, _ = orc.mx_cast(x, f, 0)
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    blocks = np.abs(xf).reshape(-1, 32).max(axis=1)
    scaled = blocks * 2.0 ** -(e8.reshape(-1).astype(np.int64) - 127)
    assert np.all((scaled >= 2.0 ** EMAX[f]) & (scaled < 2.0 ** (EMAX[f] + 1)))


@pytest.mark.parametrize("f", [0, 1])
def test_headroom_removes_clipping(f, orc):
    """One extra bit of exponent headroom: zero clipped for any finite input
    whose block exponent is not clamped; the OCP rule clips on the same
    tanh-like data (values piled up just under 1.0)."""
    rng = np.random.default_rng(22)
    x = _bf16(np.tanh(rng.standard_normal((128, 512)) * 2.0))
    _, _, clipped_ocp = orc.mx_cast(x, f, 0)
    _, _, clipped_h1 = orc.mx_cast(x, f, 1)
    assert clipped_h1 == 0
    if f == 0:
        assert clipped_ocp > 0


def test_mx_spec_vs_c_small(orc):
    """Exact specification and C oracle agree byte for byte on small
    tensors with zeros, subnormals, NaN/Inf blocks and huge blocks."""
    rng = np.random.default_rng(23)
    x = rng.standard_normal((6, 64)) * np.exp(rng.uniform(-30, 30, size=(6, 1)))
    x[0, :32] = 0.0
    x[0, 3] = -0.0
    x[1, 5] = np.nan
    x[2, 40] = -np.inf
    x[3, :32] *= 1e-38                      # bf16 subnormals
    x[4, 32:] = 3e38
    xb = _bf16(x)
    vals = [spec.bf16_bits_exact(int(b)) for b in xb.reshape(-1)]
    for f, sf in ((0, spec.E4M3), (1, spec.E5M2)):
        for h in (0, 1, 2):
            q, e8, clipped = orc.mx_cast(xb, f, h)
            qs, e8s, clipped_s = spec.mx_cast_tensor(sf, vals, 64, h)
            assert list(q.reshape(-1)) == qs
            assert list(e8.reshape(-1)) == e8s
            assert clipped == clipped_s
    q, e8, _ = orc.mx_cast(xb, 0, 0)
    assert e8[0, 0] == 0 and np.all(q[0, :32] & 0x7F == 0) and q[0, 3] == 0x80
    assert e8[1, 0] == 0xFF and np.all(q[1, :32] & 0x7F == 0x7F)
    assert e8[2, 1] == 0xFF


def test_mx_layout_row_blocks(orc):
    """Blocks run along the last dimension: permuting whole blocks of a row
    permutes the E8M0 bytes the same way; transposing does not commute."""
    rng = np.random.default_rng(24)
    x = _bf16(rng.standard_normal((4, 128)) * np.array([[1], [100], [1e-3], [7]]))
    q, e8, _ = orc.mx_cast(x, 0, 0)
    perm = [2, 0, 3, 1]
    xp = x.reshape(4, 4, 32)[:, perm, :].reshape(4, 128)
    qp, e8p, _ = orc.mx_cast(xp, 0, 0)
    assert np.array_equal(e8p, e8[:, perm])
    assert np.array_equal(qp.reshape(4, 4, 32), q.reshape(4, 4, 32)[:, perm, :])


# ---------------------------------------------------------------------------
# scale-rounding rules and column-wise blocks ("The part I would rather not
# write": NVIDIA's MXFP8 recipe rounds the shared scale up; floor, ceil and
# nearest rounding compared)
# ---------------------------------------------------------------------------

FMAX = {0: 448, 1: 57344}


def _floor_log2(r: Fraction) -> int:
    k = r.numerator.bit_length() - r.denominator.bit_length()
    if Fraction(2) ** k > r:
        k -= 1
    elif Fraction(2) ** (k + 1) <= r:
        k += 1
    return k


@pytest.mark.parametrize("f", [0, 1])
def test_mx_ceil_rule_all_bf16_amax(f, orc):
    """ceil: E = ceil(log2(A / fmax)) (exact rationals), so the scaled block
    max lands in (fmax/2, fmax] and never clips."""
    fmax = Fraction(FMAX[f])
    for b in range(1, 0x7F80):
        a = spec.f32_bits_exact(b << 16)[1]
        r = a / fmax
        k = _floor_log2(r)
        want = k if r == Fraction(2) ** k else k + 1
        want = max(-127, min(127, want))
        got = orc.mx_exp_rule(b << 16, f, 1, 0)
        assert got == want, hex(b)
        if -127 < got < 127:
            scaled = a / Fraction(2) ** got
            assert fmax / 2 < scaled <= fmax
        if b % 89 == 0:
            assert spec.mx_exp_rule([spec.E4M3, spec.E5M2][f], a, 1, 0) == want


@pytest.mark.parametrize("f", [0, 1])
def test_mx_nearest_rule_all_bf16_amax(f, orc):
    """nearest: E minimises |log2(A / fmax) - E|, checked with floating-point
    logarithms (never close to a half-way point for bf16 amax values), so the
    scaled block max lands in [fmax/sqrt2, fmax*sqrt2)."""
    fmax = FMAX[f]
    for b in range(1, 0x7F80):
        a = float(spec.f32_bits_exact(b << 16)[1])
        l = math.log2(a) - math.log2(fmax)
        cand = sorted(range(math.floor(l) - 1, math.floor(l) + 3), key=lambda e: abs(l - e))
        assert abs(abs(l - cand[0]) - abs(l - cand[1])) > 1e-9
        want = max(-127, min(127, cand[0]))
        got = orc.mx_exp_rule(b << 16, f, 2, 0)
        assert got == want, hex(b)
        if -127 < got < 127:
            scaled = a * 2.0 ** -got
            assert fmax / math.sqrt(2) <= scaled < fmax * math.sqrt(2)
        if b % 89 == 0:
            assert spec.mx_exp_rule([spec.E4M3, spec.E5M2][f], Fraction(a), 2, 0) == want


@pytest.mark.parametrize("f", [0, 1])
def test_mx_ceil_never_clips(f, orc):
    rng = np.random.default_rng(25)
    x = _bf16(np.tanh(rng.standard_normal((64, 256)) * 2.0) * np.exp(rng.uniform(-10, 10, (64, 1))))
    for axis in (0, 1):
        _, _, clipped = orc.mx_cast_ex(x, f, 1, 0, axis)
        assert clipped == 0


def test_mx_rules_spec_vs_c(orc):
    rng = np.random.default_rng(26)
    rows, cols = 64, 64
    v = rng.standard_normal((rows, cols)) * np.exp(rng.uniform(-30, 30, size=(rows, 1)))
    v[0, :] = 0.0
    v[1, 3] = np.nan
    v[40, 7] = -np.inf
    v[5, :] *= 1e-38
    xb = _bf16(v)
    vals = [spec.bf16_bits_exact(int(b)) for b in xb.reshape(-1)]
    for f, sf in ((0, spec.E4M3), (1, spec.E5M2)):
        for rule in (0, 1, 2):
            for axis in (0, 1):
                q, e8, clipped = orc.mx_cast_ex(xb, f, rule, 1 if rule == 2 else 0, axis)
                qs, e8s, cs = spec.mx_cast_tensor_ex(sf, vals, rows, cols, rule, 1 if rule == 2 else 0, axis)
                assert list(q.reshape(-1)) == qs, (f, rule, axis)
                assert list(e8.reshape(-1)) == e8s, (f, rule, axis)
                assert clipped == cs


def test_mx_colwise_is_rowwise_of_the_transpose(orc):
    """Column-wise blocks of X are the row-wise blocks of X^T."""
    rng = np.random.default_rng(27)
    x = _bf16(rng.standard_normal((96, 64)) * np.exp(rng.uniform(-5, 5, size=(1, 64))))
    for rule in (0, 1, 2):
        qc, ec, cc = orc.mx_cast_ex(x, 0, rule, 0, 1)
        qr, er, cr = orc.mx_cast_ex(np.ascontiguousarray(x.T), 0, rule, 0, 0)
        assert np.array_equal(qc, qr.T) and np.array_equal(ec, er.T) and cc == cr


def test_mx_floor_rule_matches_ocp_entry(orc):
    rng = np.random.default_rng(28)
    x = _bf16(np.tanh(rng.standard_normal((32, 128)) * 2))
    for h in (0, 1):
        q1, e1, c1 = orc.mx_cast(x, 0, h)
        q2, e2, c2 = orc.mx_cast_ex(x, 0, 0, h, 0)
        assert np.array_equal(q1, q2) and np.array_equal(e1, e2) and c1 == c2


@pytest.mark.parametrize("f", [0, 1])
def test_clip_free_rules_never_clip_any_bf16_block_max(f, orc):
    """Every positive finite bf16 value A as a block maximum (the block holds
    A, -A and 30 values in [0, A]): the round-up rule, and one or two binades
    of headroom under every rule, clip nothing, while the OCP rule without
    headroom does clip on the same blocks.  The kernels rely on this to run
    clip-free casts without a clip count."""
    a = np.arange(1, 0x7F80, dtype=np.uint32)             # bf16 bit patterns of every positive finite value
    rng = np.random.default_rng(31)
    amax = (a << 16).view(np.float32).astype(np.float64)
    rest = amax[:, None] * rng.uniform(0.0, 1.0, size=(a.size, 30))
    blocks = np.concatenate([amax[:, None], -amax[:, None], rest], axis=1)
    x = _bf16(blocks)
    assert np.array_equal(x[:, 0], a.astype(np.uint16))    # the maxima are exact
    for rule, h in ((1, 0), (1, 1), (0, 1), (2, 1), (0, 2), (2, 2)):
        _, _, clipped = orc.mx_cast_ex(x, f, rule, h, 0)
        assert clipped == 0, (rule, h)
    _, _, clipped_ocp = orc.mx_cast_ex(x, f, 0, 0, 0)
    assert clipped_ocp > 0

"""Exact-arithmetic specification of the scaled FP8 cast (second oracle).

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
benchmark's CPU-baseline leg may import anything under ``oracle/``; the
product library never does.

Every value here is a ``fractions.Fraction`` carried with an explicit sign bit,
because a Fraction has no negative zero -- the very mistake the exhaustive
format check on "what actually breaks low precision training" ("First,
catching myself") caught in its author's own exact reference.  Nothing here
uses binary floating point; it is slow and meant for small inputs.

Formats ("Mixed Precision FP16/BF16/FP8" mind-map card): a generic minifloat
with E exponent bits, M mantissa bits and bias 2^(E-1)-1, in two kinds:
IEEE (all-ones exponent = Inf/NaN; E5M2, FP16) and FN (only S.1111.111 is
NaN, no infinity; OCP E4M3, max 448).

Encoding (reading adopted where the pages are silent): the nearest point of
the format's grid extended with unbounded exponent above the largest finite
value, ties to the even significand; a rounded magnitude above the maximum
(or an infinite input) saturates to sign|max and is "clipped"; NaN maps to
sign|NaN code and is not clipped; zeros keep their sign.
"""
from __future__ import annotations

import bisect
import struct
from dataclasses import dataclass
from fractions import Fraction

INF = "inf"
NAN = "nan"


@dataclass(frozen=True)
class Minifloat:
    name: str
    ebits: int
    mbits: int
    ieee: bool

    @property
    def bias(self) -> int:
        return (1 << (self.ebits - 1)) - 1

    @property
    def nbits(self) -> int:
        return 1 + self.ebits + self.mbits

    @property
    def sign_bit(self) -> int:
        return 1 << (self.nbits - 1)

    def decode(self, code: int):
        """Return (sign, magnitude) with magnitude a Fraction, INF or NAN."""
        s = (code >> (self.nbits - 1)) & 1
        ef = (code >> self.mbits) & ((1 << self.ebits) - 1)
        mf = code & ((1 << self.mbits) - 1)
        eall = (1 << self.ebits) - 1
        if self.ieee and ef == eall:
            return s, (INF if mf == 0 else NAN)
        if not self.ieee and ef == eall and mf == (1 << self.mbits) - 1:
            return s, NAN
        if ef == 0:
            mag = Fraction(mf) * Fraction(2) ** (1 - self.bias - self.mbits)
        else:
            mag = Fraction((1 << self.mbits) + mf) * Fraction(2) ** (ef - self.bias - self.mbits)
        return s, mag

    def finite_table(self):
        """Sorted list of (magnitude, code) for every non-negative finite code."""
        out = []
        for c in range(1 << (self.nbits - 1)):
            _, m = self.decode(c)
            if isinstance(m, Fraction):
                out.append((m, c))
        out.sort()
        return out


E4M3 = Minifloat("e4m3", 4, 3, ieee=False)
E5M2 = Minifloat("e5m2", 5, 2, ieee=True)
FP16 = Minifloat("fp16", 5, 10, ieee=True)
FORMATS = {0: E4M3, 1: E5M2, 2: FP16}

_TABLES: dict = {}


def _table(fmt: Minifloat):
    if fmt.name not in _TABLES:
        tab = fmt.finite_table()
        mags = [m for m, _ in tab]
        codes = [c for _, c in tab]
        fmax = mags[-1]
        # next point of the grid extended above the maximum: one step of the
        # top binade further up; its significand parity decides ties with fmax
        top_binade = fmax.numerator.bit_length() - fmax.denominator.bit_length()
        while Fraction(2) ** top_binade > fmax:
            top_binade -= 1
        while Fraction(2) ** (top_binade + 1) <= fmax:
            top_binade += 1
        step = Fraction(2) ** (top_binade - fmt.mbits)
        over = fmax + step
        over_sig = over / step          # integer significand on that grid
        if over >= Fraction(2) ** (top_binade + 1):   # carried into next binade
            over_sig = over / (step * 2)
        _TABLES[fmt.name] = (mags, codes, fmax, over, int(over_sig) % 2 == 0)
    return _TABLES[fmt.name]


def max_code(fmt: Minifloat) -> int:
    mags, codes, *_ = _table(fmt)
    return codes[-1]


def nan_code(fmt: Minifloat) -> int:
    """The positive NaN code used for NaN results: all ones below the sign for
    the FP8 formats, the quiet NaN 0x7E00 for FP16."""
    if fmt is FP16:
        return 0x7E00
    return (1 << (fmt.nbits - 1)) - 1


def encode(fmt: Minifloat, sign: int, mag):
    """Encode sign * mag (mag: Fraction >= 0, INF or NAN). Returns (code, clipped)."""
    sb = fmt.sign_bit if sign else 0
    if mag == NAN:
        return sb | nan_code(fmt), False
    if mag == INF:
        return sb | max_code(fmt), True
    mags, codes, fmax, over, over_even = _table(fmt)
    if mag == 0:
        return sb, False
    if mag > over:
        return sb | max_code(fmt), True
    i = bisect.bisect_left(mags, mag)
    # candidates: mags[i-1] <= mag <= mags[i]  (or over when past fmax)
    lo_m, lo_c = mags[i - 1], codes[i - 1]
    if i < len(mags):
        hi_m, hi_c, hi_even, hi_over = mags[i], codes[i], codes[i] % 2 == 0, False
    else:
        hi_m, hi_c, hi_even, hi_over = over, None, over_even, True
    if mag == hi_m:
        pick_hi = True
    elif mag - lo_m < hi_m - mag:
        pick_hi = False
    elif mag - lo_m > hi_m - mag:
        pick_hi = True
    else:                                   # tie: even significand wins
        pick_hi = hi_even
    if pick_hi and hi_over:
        return sb | max_code(fmt), True
    return sb | (hi_c if pick_hi else lo_c), False


# ---------------------------------------------------------------------------
# IEEE inputs (bf16 / fp32 bit patterns) as exact values
# ---------------------------------------------------------------------------

def f32_bits_exact(bits: int):
    """fp32 bit pattern -> (sign, Fraction | INF | NAN)."""
    s = (bits >> 31) & 1
    ef = (bits >> 23) & 0xFF
    mf = bits & 0x7FFFFF
    if ef == 0xFF:
        return s, (INF if mf == 0 else NAN)
    if ef == 0:
        return s, Fraction(mf) * Fraction(2) ** -149
    return s, Fraction(mf | 0x800000) * Fraction(2) ** (ef - 150)


def bf16_bits_exact(bits: int):
    return f32_bits_exact(bits << 16)


def f32_of_double(v: float) -> int:
    return struct.unpack("<I", struct.pack("<f", v))[0]


def cast(fmt: Minifloat, sign: int, mag, e: int):
    """Scaled cast: q = sat-RNE(x * 2^e)."""
    if isinstance(mag, Fraction):
        mag = mag * Fraction(2) ** e
    return encode(fmt, sign, mag)


# ---------------------------------------------------------------------------
# Per-tensor policy pieces ("Practice c06/E3, worked solution")
# ---------------------------------------------------------------------------

def fmax_of(fmt: Minifloat) -> Fraction:
    return _table(fmt)[2]


def scale_exp(fmt: Minifloat, amax: Fraction, margin: int):
    """Largest integer e in [-126, 126] with 2^e * amax <= fmax * 2^-margin.

    Returns None when amax is zero (the caller keeps its previous exponent).
    """
    if amax == 0:
        return None
    limit = fmax_of(fmt) * Fraction(2) ** -margin
    # start from a bound and walk: the definition, checked step by step
    e = 126
    while e > -126 and Fraction(2) ** e * amax > limit:
        e -= 1
    return e


def mx_exp(fmt: Minifloat, amax: Fraction, headroom: int) -> int:
    """OCP shared exponent: floor(log2 amax) - emax_elem (+ headroom),
    clamped to [-127, 127]; a zero block gives -127."""
    if amax == 0:
        return -127
    p = 0
    while Fraction(2) ** (p + 1) <= amax:
        p += 1
    while Fraction(2) ** p > amax:
        p -= 1
    fmax = fmax_of(fmt)
    emax = 0
    while Fraction(2) ** (emax + 1) <= fmax:
        emax += 1
    return max(-127, min(127, p - emax + headroom))


# ---------------------------------------------------------------------------
# Arithmetic on format values with IEEE signed-zero rules (for the exhaustive
# product / sum check of "First, catching myself")
# ---------------------------------------------------------------------------

def mul(a, b):
    """(sign, mag) x (sign, mag) -> (sign, mag) exactly, zero keeps its sign."""
    (sa, ma), (sb, mb) = a, b
    s = sa ^ sb
    if ma == NAN or mb == NAN:
        return 0, NAN
    if ma == INF or mb == INF:
        if ma == 0 or mb == 0:
            return 0, NAN
        return s, INF
    return s, ma * mb


def add(a, b):
    """(sign, mag) + (sign, mag) under round-to-nearest signed-zero rules:
    an exact zero sum is +0 unless both operands are zeros of sign 1."""
    (sa, ma), (sb, mb) = a, b
    if ma == NAN or mb == NAN:
        return 0, NAN
    if ma == INF or mb == INF:
        if ma == INF and mb == INF and sa != sb:
            return 0, NAN
        return (sa, INF) if ma == INF else (sb, INF)
    va = -ma if sa else ma
    vb = -mb if sb else mb
    v = va + vb
    if v == 0:
        if ma == 0 and mb == 0 and sa == 1 and sb == 1:
            return 1, Fraction(0)
        return 0, Fraction(0)
    return (1 if v < 0 else 0), abs(v)


# ---------------------------------------------------------------------------
# Small-tensor reference (pure Python loops; tiny inputs only)
# ---------------------------------------------------------------------------

def tensor_amax(vals):
    """vals: list of (sign, mag).  Exact max |x| with NaN > Inf > finite."""
    best = Fraction(0)
    for _, m in vals:
        if m == NAN:
            return NAN
        if m == INF:
            best = INF
        elif best != INF and m > best:
            best = m
    return best


def cast_tensor(fmt, vals, e):
    out, clipped = [], 0
    for s, m in vals:
        c, cl = cast(fmt, s, m, e)
        out.append(c)
        clipped += int(cl)
    return out, clipped


def mx_cast_tensor(fmt, vals, cols, headroom):
    """vals row-major, 32-element blocks along the last dimension."""
    assert cols % 32 == 0
    q, e8, clipped = [], [], 0
    for b in range(len(vals) // 32):
        blk = vals[32 * b: 32 * b + 32]
        a = tensor_amax(blk)
        if a in (NAN, INF):
            e8.append(0xFF)
            q.extend(fmt.sign_bit * s | nan_code(fmt) for s, _ in blk)
            continue
        E = mx_exp(fmt, a, headroom)
        e8.append(E + 127)
        for s, m in blk:
            c, cl = cast(fmt, s, m, -E)
            q.append(c)
            clipped += int(cl)
    return q, e8, clipped


def error_stats(fmt, vals, codes, scale_of_index):
    """Exact mean squared error and mean error (bias) of deq - x over the
    elements with finite input; scale_of_index(i) gives deq's power-of-two
    factor as a Fraction (None: skip the element)."""
    sq, sm, k = Fraction(0), Fraction(0), 0
    for i, ((s, m), c) in enumerate(zip(vals, codes)):
        if m in (NAN, INF):
            continue
        sc = scale_of_index(i)
        if sc is None:
            continue
        cs, cm = fmt.decode(int(c))
        deq = (-cm if cs else cm) * sc
        x = -m if s else m
        d = deq - x
        sq += d * d
        sm += d
        k += 1
    if k == 0:
        return Fraction(0), Fraction(0), 0
    return sq / k, sm / k, k


# ---------------------------------------------------------------------------
# MX scale-rounding rules and block direction (see oracle.c for the readings:
# 0 OCP floor, 1 smallest E with A 2^-E <= fmax, 2 E nearest log2(A / fmax))
# ---------------------------------------------------------------------------

def mx_exp_rule(fmt: Minifloat, amax: Fraction, rule: int, headroom: int) -> int:
    if rule == 0:
        return mx_exp(fmt, amax, headroom)
    if amax == 0:
        return -127
    fmax = fmax_of(fmt)
    e = -200
    while amax / Fraction(2) ** e > fmax:
        e += 1
    if rule == 2:
        # keep e when fmax / (A 2^-e) <= (A 2^-(e-1)) / fmax, else e - 1
        lo = fmax / (amax / Fraction(2) ** e)
        hi = (amax / Fraction(2) ** (e - 1)) / fmax
        if not lo <= hi:
            e -= 1
    return max(-127, min(127, e + headroom))


def mx_cast_tensor_ex(fmt, vals, rows, cols, rule, headroom, axis):
    """vals row-major [rows, cols]; returns (q list row-major, e8m0 list in
    its own row-major layout, clipped)."""
    q = [None] * (rows * cols)
    if axis == 0:
        blocks = [[r * cols + c0 + j for j in range(32)] for r in range(rows) for c0 in range(0, cols, 32)]
    else:
        blocks = [[(r0 + j) * cols + c for j in range(32)] for r0 in range(0, rows, 32) for c in range(cols)]
    e8, clipped = [], 0
    for idx in blocks:
        blk = [vals[i] for i in idx]
        a = tensor_amax(blk)
        if a in (NAN, INF):
            e8.append(0xFF)
            for i, (s, _) in zip(idx, blk):
                q[i] = fmt.sign_bit * s | nan_code(fmt)
            continue
        E = mx_exp_rule(fmt, a, rule, headroom)
        e8.append(E + 127)
        for i, (s, m) in zip(idx, blk):
            c, cl = cast(fmt, s, m, -E)
            q[i] = c
            clipped += int(cl)
    return q, e8, clipped


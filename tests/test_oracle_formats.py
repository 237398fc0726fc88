"""Pins of the oracle's number formats against the pages and against
independent library routines (numpy float16, torch float8, ml_dtypes).

Formats: "Mixed Precision FP16/BF16/FP8" mind-map card, bit layouts and ranges.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import spec

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FMT = {"e4m3": 0, "e5m2": 1, "fp16": 2}
SPECFMT = {"e4m3": spec.E4M3, "e5m2": spec.E5M2, "fp16": spec.FP16}


def _exact(s: str) -> Fraction:
    """Parse '65504', '2^-14', '2^15*(2-2^-10)'."""
    s = s.replace("^", "**")
    return Fraction(eval(s, {"__builtins__": {}}, {})) if "**" in s else Fraction(s)


def _golden_constants():
    rows = []
    with open(os.path.join(GOLDEN, "format_constants.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append(line.split()[:3])
    return rows


def _finite_positive(fmt_name, orc):
    n = 1 << (SPECFMT[fmt_name].nbits - 1)
    vals = [orc.decode(FMT[fmt_name], c) for c in range(n)]
    return [v for v in vals if math.isfinite(v) and v > 0]


@pytest.mark.parametrize("row", _golden_constants(), ids=lambda r: f"{r[0]}-{r[1]}")
def test_printed_constants(row, orc):
    """Every printed constant is reproduced by the generic codec (C) and the
    exact specification."""
    fmt_name, qty, val = row
    if fmt_name == "bf16":                       # 1+8+7: the upper half of fp32
        assert val == "1+8+7"
        b = spec.f32_bits_exact(0x7F7F0000)      # largest finite bf16
        assert b[1] == Fraction(2) ** 127 * (2 - Fraction(2) ** -7)
        return
    sf = SPECFMT[fmt_name]
    if qty == "layout":
        assert val == f"1+{sf.ebits}+{sf.mbits}"
        return
    pos = _finite_positive(fmt_name, orc)
    exact_pos = sorted(m for c in range(1 << (sf.nbits - 1))
                       for s, m in [sf.decode(c)] if isinstance(m, Fraction) and m > 0)
    if qty in ("max", "max_formula"):
        got_c, got_s = max(pos), exact_pos[-1]
    elif qty == "min_normal":
        got_c = min(v for v in pos if v >= 2.0 ** (1 - sf.bias))
        got_s = min(m for m in exact_pos if m >= Fraction(2) ** (1 - sf.bias))
        assert got_c == 2.0 ** (1 - sf.bias)     # and it is the smallest normal
    elif qty == "min_subnormal":
        got_c, got_s = min(pos), exact_pos[0]
    else:
        raise AssertionError(qty)
    assert Fraction(got_c) == _exact(val)
    assert got_s == _exact(val)


def test_fp16_all_codes_match_numpy(orc):
    """The generic minifloat at (5, 10, IEEE) decodes all 65,536 codes exactly
    like numpy's float16."""
    codes = np.arange(65536, dtype=np.uint32)
    ref = codes.astype(np.uint16).view(np.float16).astype(np.float64)
    got = np.array([orc.decode(2, int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))   # -0 kept


def test_fp16_encode_matches_numpy(orc):
    """The generic encoder at FP16 rounds like numpy's float64->float16 (RNE)
    on in-range values, including ties and subnormals."""
    rng = np.random.default_rng(1)
    v = np.concatenate([
        rng.standard_normal(20000) * 100.0,
        rng.standard_normal(5000) * 1e-6,                       # subnormals
        np.arange(-2048, 2049) * 2.0 ** -25,                     # ties at 2^-25
        (np.arange(1024, 2048) + 0.5) * 2.0 ** -9,               # ties in [1,2)
        [65504.0, -65504.0, 65519.0, 0.0, -0.0],
    ])
    ref = v.astype(np.float16).view(np.uint16)
    for x, r in zip(v, ref):
        code, clipped = orc.encode_double(2, float(x))
        assert code == int(r), (x, hex(code), hex(int(r)))
        assert not clipped


@pytest.mark.parametrize("fmt_name,tdt", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_fp8_all_codes_match_torch(fmt_name, tdt, orc):
    """All 256 codes decode like torch's float8 types (a library routine),
    and like the exact specification."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(tdt).to(torch.float64).numpy()
    sf = SPECFMT[fmt_name]
    for c in range(256):
        got = orc.decode(FMT[fmt_name], c)
        s, m = sf.decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got) and m == spec.NAN
            continue
        assert got == ref[c] and math.copysign(1, got) == math.copysign(1, ref[c]), c
        if m == spec.INF:
            assert math.isinf(got) and (got < 0) == bool(s)
        else:
            assert Fraction(abs(got)) == m and (math.copysign(1, got) < 0) == bool(s)


@pytest.mark.parametrize("fmt_name", ["e4m3", "e5m2"])
def test_fp8_all_codes_match_ml_dtypes(fmt_name, orc):
    ml = pytest.importorskip("ml_dtypes")
    dt = ml.float8_e4m3fn if fmt_name == "e4m3" else ml.float8_e5m2
    ref = np.arange(256, dtype=np.uint8).view(dt).astype(np.float64)
    got = np.array([orc.decode(FMT[fmt_name], c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_fp8_specials():
    """Special codes of the two OCP formats."""
    assert spec.E4M3.decode(0x7F)[1] == spec.NAN and spec.E4M3.decode(0xFF)[1] == spec.NAN
    assert spec.E4M3.decode(0x7E)[1] == 448 and spec.E4M3.decode(0x78)[1] == 256
    assert spec.E4M3.decode(0x08)[1] == Fraction(2) ** -6      # min normal
    assert spec.E4M3.decode(0x01)[1] == Fraction(2) ** -9      # min subnormal
    assert spec.E5M2.decode(0x7C) == (0, spec.INF) and spec.E5M2.decode(0xFC) == (1, spec.INF)
    for c in (0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF):
        assert spec.E5M2.decode(c)[1] == spec.NAN
    assert spec.E5M2.decode(0x7B)[1] == 57344
    assert spec.E5M2.decode(0x04)[1] == Fraction(2) ** -14
    assert spec.E5M2.decode(0x01)[1] == Fraction(2) ** -16


@pytest.mark.parametrize("fmt_name", ["e4m3", "e5m2"])
def test_roundtrip_every_code(fmt_name, orc):
    """encode(decode(c)) == c for every non-NaN code, including both zeros;
    infinities (E5M2) saturate to the largest finite code and clip."""
    sf = SPECFMT[fmt_name]
    for c in range(256):
        s, m = sf.decode(c)
        if m == spec.NAN:
            continue
        v = orc.decode(FMT[fmt_name], c)
        code_c, cl_c = orc.encode_double(FMT[fmt_name], v)
        code_s, cl_s = spec.encode(sf, s, m)
        if m == spec.INF:
            want = (0x80 if s else 0) | spec.max_code(sf)
            assert (code_c, cl_c) == (want, True) and (code_s, cl_s) == (want, True)
        else:
            assert (code_c, cl_c) == (c, False) and (code_s, cl_s) == (c, False)


@pytest.mark.parametrize("fmt_name,fmax,over", [("e4m3", 448.0, 464.0), ("e5m2", 57344.0, 61440.0)])
def test_saturation_boundary(fmt_name, fmax, over, orc):
    """The top of the range: the tie between the maximum and the next point of
    the extended grid goes to the even significand (448 for E4M3, so 464 does
    not clip; 65536 for E5M2, so 61440 clips)."""
    f = FMT[fmt_name]
    up = float(np.nextafter(np.float32(over), np.float32(np.inf)))
    down = float(np.nextafter(np.float32(over), np.float32(0)))
    mx = 0x7E if f == 0 else 0x7B
    assert orc.encode_double(f, fmax) == (mx, False)
    assert orc.encode_double(f, down) == (mx, False)
    assert orc.encode_double(f, up) == (mx, True)
    assert orc.encode_double(f, over) == (mx, f == 1)
    assert orc.encode_double(f, -up) == (0x80 | mx, True)
    assert orc.encode_double(f, float("inf")) == (mx, True)
    assert orc.encode_double(f, float("-inf")) == (0x80 | mx, True)
    code, cl = orc.encode_double(f, float("nan"))
    assert code == 0x7F and not cl
    sf = SPECFMT[fmt_name]
    assert spec.encode(sf, 0, Fraction(over)) == (mx, f == 1)
    assert spec.encode(sf, 0, Fraction(up)) == (mx, True)


def _signed_zero_rows():
    rows = []
    with open(os.path.join(GOLDEN, "signed_zero.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append(line.split())
    return rows


@pytest.mark.parametrize("row", _signed_zero_rows(), ids=lambda r: "-".join(r[:3]))
def test_signed_zero(row, orc):
    op, fmt_name, a, b, want = row
    f, sf, want = FMT[fmt_name], SPECFMT[fmt_name], int(want, 16)
    a = float(a)
    if op == "cast":
        xb = spec.f32_of_double(a)
        assert orc.cast_scalar(f, xb, 0)[0] == want
        s, m = spec.f32_bits_exact(xb)
        assert spec.cast(sf, s, m, 0)[0] == want
        return
    b = float(b)
    va = (1 if math.copysign(1, a) < 0 else 0, Fraction(abs(a)))
    vb = (1 if math.copysign(1, b) < 0 else 0, Fraction(abs(b)))
    r_c = a * b if op == "mul" else a + b
    r_s = spec.mul(va, vb) if op == "mul" else spec.add(va, vb)
    assert orc.encode_double(f, r_c)[0] == want
    assert spec.encode(sf, *r_s)[0] == want


def _all_bf16_as_f32():
    b = np.arange(65536, dtype=np.uint32) << 16
    return b.astype(np.uint32)


@pytest.mark.parametrize("fmt_name,tdt", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_cast_all_bf16_times_scales_matches_torch(fmt_name, tdt, orc):
    """Every bf16 value times 2^e for e in -30..30 (step 3), cast by the C
    oracle, equals torch's float8 RNE conversion wherever the scaled value is
    within the format's range (torch does not saturate beyond it)."""
    f = FMT[fmt_name]
    fmax = 448.0 if f == 0 else 57344.0
    xb = _all_bf16_as_f32()
    with np.errstate(invalid="ignore"):
        xf = xb.view(np.float32).astype(np.float64)
    for e in range(-30, 31, 3):
        q, _, _ = orc.cast(xb, f, e)
        v = xf * 2.0 ** e
        ok = np.isfinite(v) & (np.abs(v) <= fmax)
        ref = torch.from_numpy(v[ok]).to(torch.float32).to(tdt).view(torch.uint8).numpy()
        assert np.array_equal(q[ok], ref), e
        # beyond the range every value lands on sign|max (rounded or saturated)
        big = np.isfinite(v) & (np.abs(v) > fmax)
        mx = 0x7E if f == 0 else 0x7B
        want = np.where(v[big] < 0, 0x80, 0) | mx
        assert np.array_equal(q[big], want.astype(np.uint8)), e
        nan = np.isnan(xf)
        assert np.all((q[nan] & 0x7F) == 0x7F)
        assert np.array_equal(q[nan] >> 7, (xb[nan] >> 31).astype(np.uint8))

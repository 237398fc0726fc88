"""Oracle model of one tensor's scaling state across training steps.

TEST INFRASTRUCTURE ONLY (tests, smoke check, benchmark CPU baseline).

Follows "Practice c06/E3, worked solution": the statistic is the largest |x|
of the tensor, watched over a window of steps; the scale is the largest power
of two keeping that window maximum at or below the format's largest finite
value divided by 2^margin; the previous scale is kept under a hysteresis rule.
The gist.science summary of "Max-Window Scale Estimation for Near-Lossless HiF8
W8A8 QAT" (Methodology, "Amax algorithms") names the variants: most-recent
(window 1), max over a history window (64 there), and current tensor scaling.

Estimators ("Amax algorithms" of the summary; "recompute the scale every
fixed number of steps" of the worked solution):
  * max-window (default): the statistic is the largest amax of the window;
  * exponential smoothing: the statistic is a running average of the amax,
    avg <- avg + alpha * (amax - avg) evaluated in fp32 (three roundings, no
    fused multiply-add), started at the first cast's amax; a non-finite amax
    does not enter the average;
  * recompute interval k: the exponent is recomputed only when the number
    of earlier casts is a multiple of k, and kept otherwise.

Readings adopted where the pages are silent:
  * the window holds the amaxes of the W steps *before* this one; this step's
    amax enters it after the cast;
  * an empty window (first step, or W = 0) means current scaling: the
    exponent comes from this tensor's own amax (a second pass);
  * a zero or non-finite window maximum keeps the previous exponent (0 when
    there is none);
  * hysteresis h (in binades, 0 = off): an upward move of at most h binades
    keeps the previous exponent; a downward move is always taken, so the
    no-overflow promise of the worked solution is never delayed;
  * the exponent is clamped to [-126, 126] so that 2^e and 2^-e are normal
    fp32 numbers.
"""
from __future__ import annotations

import struct

import numpy as np

from . import coracle


def f32_of_bits(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", b & 0xFFFFFFFF))[0]


def bits_of_f32(v: float) -> int:
    return struct.unpack("<I", struct.pack("<f", v))[0]


MAX_WINDOW, EMA = 0, 1


class ScalingState:
    """One tensor's history ring, previous exponent and policy."""

    def __init__(self, fmt: int, window: int, margin: int = 0, hysteresis: int = 0,
                 estimator: int = MAX_WINDOW, alpha: float = 1.0, interval: int = 1):
        self.fmt, self.window, self.margin, self.hysteresis = fmt, window, margin, hysteresis
        self.estimator, self.interval = estimator, interval
        self.alpha = np.float32(alpha)
        self.hist: list[int] = []          # amax bit patterns, oldest first
        self.prev_e: int | None = None
        self.steps = 0
        self.avg: np.float32 | None = None   # running average (smoothing estimator)

    def uses_current(self) -> bool:
        if self.estimator == EMA:
            return self.steps == 0
        return self.window == 0 or not self.hist

    def statistic(self) -> int:
        """fp32 bits of the statistic the next exponent comes from."""
        if self.estimator == EMA:
            return 0x7FC00000 if self.avg is None else bits_of_f32(float(self.avg))
        return max(self.hist)

    def exponent(self, window_amax_bits: int) -> int:
        if (self.interval > 1 and self.prev_e is not None and self.steps % self.interval != 0):
            return self.prev_e
        e_new = coracle.scale_exp(window_amax_bits, self.fmt, self.margin)
        if e_new is None:                               # zero or non-finite
            return self.prev_e if self.prev_e is not None else 0
        if (self.prev_e is not None and e_new > self.prev_e
                and e_new - self.prev_e <= self.hysteresis):
            return self.prev_e
        return e_new

    def step(self, x: np.ndarray, nthreads: int = 1):
        """Cast one step's tensor x (raw bits).  Returns
        (q, amax_bits, scale_inv_bits, clipped, e)."""
        if self.uses_current():
            a_w = coracle.amax(x, nthreads)
        else:
            a_w = self.statistic()
        e = self.exponent(a_w)
        q, a_cur, clipped = coracle.cast(x, self.fmt, e, nthreads)
        self.record(a_cur, e)
        return q, a_cur, bits_of_f32(2.0 ** -e), clipped, e

    def record(self, amax_bits: int, e: int):
        if self.estimator == EMA and (amax_bits & 0x7FFFFFFF) < 0x7F800000:
            a = np.float32(f32_of_bits(amax_bits))
            if self.avg is None:
                self.avg = a
            else:
                self.avg = np.float32(self.avg + np.float32(self.alpha * np.float32(a - self.avg)))
        if self.window > 0:
            self.hist.append(amax_bits)
            del self.hist[:-self.window]
        self.prev_e = e
        self.steps += 1


class LossScaler:
    """Dynamic loss scaling ("Mixed Precision FP16/BF16/FP8" mind-map card:
    multiply the loss by S; on Inf/NaN set S <- S/2 and skip the step; after
    a period without overflow double S).  Readings: the period is
    `growth_interval` consecutive clean steps; S stays within
    [min_scale, max_scale]; a step is non-finite when any of its casts saw a
    NaN or Inf input."""

    def __init__(self, init_scale: float, growth_interval: int,
                 min_scale: float = 1.0, max_scale: float = 2.0 ** 24):
        self.scale = np.float32(init_scale)
        self.growth_interval = growth_interval
        self.min_scale, self.max_scale = np.float32(min_scale), np.float32(max_scale)
        self.good = 0

    def update(self, nonfinite_counts) -> bool:
        """Returns True when the step must be skipped."""
        if any(int(c) > 0 for c in nonfinite_counts):
            self.scale = max(self.min_scale, np.float32(self.scale * np.float32(0.5)))
            self.good = 0
            return True
        self.good += 1
        if self.good >= self.growth_interval:
            self.scale = min(self.max_scale, np.float32(self.scale * np.float32(2.0)))
            self.good = 0
        return False


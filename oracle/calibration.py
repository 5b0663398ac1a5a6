"""Oracle calibration statistics of one K or V tensor (test infrastructure; see the package
docstring).

[SCALES §Calibration] The converter scale is the observed max envelope over 448, and the
calibration reports, per layer and tensor, max-abs, p99.9, p99.99 and saturation.
[E4M3-PR §Why calibrated scale is part of this contract] At a given scale, the share of
nonzero elements that fall below E4M3's smallest subnormal magnitude (2^-9) and the share
in the subnormal range [2^-9, 2^-6).
[E4M3-PR §Implementation scope] The statistics are per layer and per tensor.

Readings (the pages do not define the statistics further):
  * Inputs are bf16 (or fp16) values, widened exactly to fp32. Infinite and NaN inputs are
    counted apart and take part in nothing else.
  * max-abs, p99.9 and p99.99 are order statistics of |x| over the finite elements. A
    percentile is the nearest rank: with the finite magnitudes sorted ascending
    a_1 <= ... <= a_N, p_q = a_ceil(q N), q = 999/1000 or 9999/10000 taken as exact
    fractions. N = 0 gives 0.
  * The scale is the one passed in, or, when none is passed, the calibrated
    amax / 448 (fp32 IEEE division). Each finite element's scaled magnitude is
    y = |x| / scale, one fp32 IEEE division.
  * below_subnormal counts nonzero elements with y < 2^-9; subnormal counts 2^-9 <= y < 2^-6.
  * saturated counts elements that the saturating encoder clips: those whose nearest value
    on the E4M3 grid continued past 448 (the next step would be 480) lies above 448, i.e.
    y > 464 (464 itself ties to 448, the even mantissa). With the calibrated scale the
    largest element gives y = 448 up to one rounding, so it never counts, matching the
    pages' "zero observed saturation" for calibrated scales.
  * A scale of 0 (every element zero) leaves the three scaled counts at 0.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = np.float32(448.0)
MIN_SUBNORMAL = np.float32(2.0 ** -9)
MIN_NORMAL = np.float32(2.0 ** -6)
SATURATION_EDGE = np.float32(464.0)  # midpoint of 448 and 480 on the continued E4M3 grid
NUM_BINS = 1 << 15  # 16-bit magnitudes: the 15 bits below the sign


def _f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    if dtype == "f16":
        return b.view(np.float16).astype(np.float32)
    if dtype == "bf16":
        return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)
    raise ValueError(f"unknown activation type {dtype!r}")


def magnitude_histogram(x_bits: np.ndarray) -> np.ndarray:
    """Counts of each 16-bit magnitude bit pattern (bits & 0x7FFF): int64 [32768]."""
    b = np.ascontiguousarray(x_bits, dtype=np.uint16).ravel()
    return np.bincount((b & np.uint16(0x7FFF)).astype(np.int64), minlength=NUM_BINS).astype(np.int64)


def nearest_rank(sorted_values: np.ndarray, num: int, den: int):
    """a_ceil(num/den * N) of an ascending array (1-based rank, exact integer arithmetic)."""
    n = int(sorted_values.size)
    if n == 0:
        return np.float32(0.0)
    rank = -((-num * n) // den)  # ceil(num * n / den)
    return np.float32(sorted_values[max(rank, 1) - 1])


def calibration_stats(x_bits: np.ndarray, scale=None, dtype: str = "bf16") -> dict:
    """Statistics of one tensor given as bf16 (or fp16, dtype='f16') bit patterns (any shape)."""
    x = _f32(x_bits, dtype)
    finite = np.isfinite(x)
    a = np.abs(x[finite]).astype(np.float32)
    a_sorted = np.sort(a)
    amax = np.float32(a_sorted[-1]) if a_sorted.size else np.float32(0.0)
    if scale is None:
        s = np.float32(amax / E4M3_MAX)  # fp32 IEEE division
    else:
        s = np.float32(scale)
    out = {
        "count": int(a.size),
        "zeros": int(np.count_nonzero(a == 0)),
        "nonfinite": int(x.size - a.size),
        "amax": amax,
        "p99_9": nearest_rank(a_sorted, 999, 1000),
        "p99_99": nearest_rank(a_sorted, 9999, 10000),
        "scale": s,
        "below_subnormal": 0,
        "subnormal": 0,
        "saturated": 0,
    }
    if s > 0 and a.size:
        y = (a / s).astype(np.float32)  # float32 / float32: IEEE round to nearest
        out["below_subnormal"] = int(np.count_nonzero((a != 0) & (y < MIN_SUBNORMAL)))
        out["subnormal"] = int(np.count_nonzero((y >= MIN_SUBNORMAL) & (y < MIN_NORMAL)))
        out["saturated"] = int(np.count_nonzero(y > SATURATION_EDGE))
    return out

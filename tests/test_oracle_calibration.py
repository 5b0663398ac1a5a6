"""Pins of the oracle's calibration statistics (CPU only).

"Qwen3.8 Flash Next NVFP4 QSA FP8 E4M3 KV Scales" §Calibration: scale = max envelope / 448;
max-abs, p99.9, p99.99 and saturation per tensor. "[Model][SM70][FP8] Add calibrated E4M3
QSA KV cache" §Why calibrated scale is part of this contract: nonzero elements below E4M3's
minimum subnormal (2^-9) and in the subnormal range below 2^-6.

The statistics are pinned by a hand-worked fixture, numpy's own inverted-CDF quantile,
closed forms on constructed inputs, a brute-force rounding on the E4M3 grid continued past
448, and invariants (sign symmetry, histogram additivity, zero saturation at the
calibrated scale).
"""

import numpy as np
import pytest

from oracle.calibration import calibration_stats, magnitude_histogram, nearest_rank


def bits(values):
    """bf16 bit patterns of values that bf16 represents exactly (asserted)."""
    f = np.asarray(values, dtype=np.float32)
    b = (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    back = (b.astype(np.uint32) << np.uint32(16)).view(np.float32)
    assert np.array_equal(back, f, equal_nan=True), "not a bf16 value"
    return b


def test_hand_worked_fixture():
    x = bits([0.0, -0.0, 1.0, -2.0, 0.5, 2.0 ** -10, 3 * 2.0 ** -8, np.inf, np.nan, 466.0, -464.0])
    st = calibration_stats(x, scale=1.0)
    # finite magnitudes sorted: 0, 0, 2^-10, 3*2^-8, 0.5, 1, 2, 464, 466
    assert st["count"] == 9 and st["zeros"] == 2 and st["nonfinite"] == 2
    assert st["amax"] == np.float32(466.0)
    assert st["p99_9"] == np.float32(466.0) and st["p99_99"] == np.float32(466.0)  # ranks ceil(8.991) = 9
    assert st["below_subnormal"] == 1  # 2^-10 (the zeros are not counted)
    assert st["subnormal"] == 1        # 3 * 2^-8 = 0.01171875 < 2^-6
    assert st["saturated"] == 1        # 466; 464 ties to 448
    assert st["scale"] == np.float32(1.0)


def test_nearest_rank_closed_form_on_distinct_values():
    # 2000 distinct increasing bf16 magnitudes: bit patterns 0x3F80 + i
    b = (np.arange(2000) + 0x3F80).astype(np.uint16)
    vals = (b.astype(np.uint32) << 16).view(np.float32)
    rng = np.random.default_rng(3)
    st = calibration_stats(rng.permutation(b), scale=1.0)
    assert st["p99_9"] == vals[1997]   # rank ceil(0.999 * 2000) = 1998
    assert st["p99_99"] == vals[1999]  # rank ceil(1999.8) = 2000
    assert st["amax"] == vals[1999]


@pytest.mark.parametrize("n", [7, 123, 1001, 4567, 20011])
def test_nearest_rank_matches_numpy_inverted_cdf(n):
    rng = np.random.default_rng(n)
    a = np.sort(np.abs(rng.standard_normal(n)).astype(np.float32))
    for num, den in [(999, 1000), (9999, 10000), (1, 2)]:
        if (num * n) % den == 0:
            continue  # q n an integer: numpy's float q would make the rank ambiguous
        ref = np.quantile(a, num / den, method="inverted_cdf")
        assert nearest_rank(a, num, den) == np.float32(ref)


def test_percentiles_are_of_magnitudes_and_sign_symmetric():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(30000) * 3).astype(np.float32)
    b = (x.view(np.uint32) >> 16).astype(np.uint16)
    s1 = calibration_stats(b)
    s2 = calibration_stats(b ^ np.uint16(0x8000))
    assert s1 == s2
    a = np.sort(np.abs((b.astype(np.uint32) << 16).view(np.float32)))
    # at least 99.9 % of the magnitudes are <= p99.9 and fewer than that are below it
    assert np.count_nonzero(a <= s1["p99_9"]) >= 0.999 * a.size > np.count_nonzero(a < s1["p99_9"])


@pytest.mark.parametrize("scale", [1.0, 0.5, 0.0171247218, 3.0])
def test_subnormal_band_edges(scale):
    s = np.float32(scale)
    # the bf16 neighbours of the two band edges times the scale, each classified by hand
    lo, hi = np.float32(2.0 ** -9), np.float32(2.0 ** -6)
    cand = []
    for edge in (lo, hi):
        t = np.float32(edge * s)
        tb = (t.view(np.uint32) >> 16).astype(np.uint16)
        cand += [tb - 1, tb, tb + 1]
    b = np.array(cand, dtype=np.uint16)
    st = calibration_stats(b, scale=s)
    y = ((b.astype(np.uint32) << 16).view(np.float32) / s).astype(np.float32)
    assert st["below_subnormal"] == sum(1 for v in y if 0 < v < lo)
    assert st["subnormal"] == sum(1 for v in y if lo <= v < hi)


def _nearest_on_continued_grid(y: float) -> float:
    """Round y > 0 to the E4M3 grid continued past 448 (2^e (1 + m/8)), ties to even m."""
    e = int(np.floor(np.log2(y)))
    step = 2.0 ** (e - 3)
    lo = np.floor(y / step) * step
    hi = lo + step
    if y - lo < hi - y:
        return lo
    if hi - y < y - lo:
        return hi
    m_lo = int(round(lo / 2.0 ** e * 8)) - 8
    return lo if m_lo % 2 == 0 else hi


def test_saturation_edge_by_brute_force_rounding():
    # every bf16 value in [400, 520] at scale 1: saturated <=> its nearest continued-grid
    # value lies above 448
    b = np.arange(0x43C8, 0x4403, dtype=np.uint16)
    vals = (b.astype(np.uint32) << 16).view(np.float32)
    assert vals[0] == 400.0 and vals[-1] == 520.0
    expect = sum(1 for v in vals if _nearest_on_continued_grid(float(v)) > 448.0)
    assert expect > 0
    assert calibration_stats(b, scale=1.0)["saturated"] == expect


def test_calibrated_scale_never_saturates():
    rng = np.random.default_rng(9)
    for trial in range(20):
        x = rng.standard_normal(5000).astype(np.float32) * np.float32(rng.uniform(0.01, 50))
        x[rng.choice(5000, 50, replace=False)] *= np.float32(16.0)
        b = (x.view(np.uint32) >> 16).astype(np.uint16)
        st = calibration_stats(b)
        assert st["saturated"] == 0
        assert st["scale"] == np.float32(st["amax"] / np.float32(448.0))


def test_zero_tensor_and_empty():
    st = calibration_stats(np.zeros(10, dtype=np.uint16))
    assert st["scale"] == 0 and st["amax"] == 0 and st["zeros"] == 10
    assert st["below_subnormal"] == st["subnormal"] == st["saturated"] == 0
    st = calibration_stats(np.zeros(0, dtype=np.uint16), scale=1.0)
    assert st["count"] == 0 and st["p99_9"] == 0


def test_histogram_counts_and_additivity():
    rng = np.random.default_rng(11)
    a = rng.integers(0, 1 << 16, 5000).astype(np.uint16)
    b = rng.integers(0, 1 << 16, 3000).astype(np.uint16)
    ha, hb = magnitude_histogram(a), magnitude_histogram(b)
    assert ha.sum() == 5000 and ha.shape == (32768,)
    assert np.array_equal(magnitude_histogram(np.concatenate([a, b])), ha + hb)
    u, c = np.unique(a & 0x7FFF, return_counts=True)
    assert np.array_equal(ha[u], c) and ha.sum() == c.sum()

"""Pins for the oracle's E4M3 decoder/encoder (CPU only).

The format facts come from "Qwen3.8 Flash Next NVFP4 QSA FP8 E4M3 KV Scales" §Calibration
(448 = largest finite magnitude) and "[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache"
§Why calibrated scale is part of this contract (2^-9 smallest subnormal, 2^-6 boundary);
"[Perf][SM70][FP8] Hoist QSA E4M3 KV scales" §AWQ formal-r6 replication reports a suite over
all 256 encodings, which the exhaustive checks here mirror.
"""

import math
import os

import numpy as np
import pytest
import torch

from oracle import quant

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_encode.txt")


def _golden():
    out = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            y, code = line.split()
            out.append((float(y), int(code, 16)))
    return out


def test_decode_all_256_against_torch_float8():
    codes = np.arange(256, dtype=np.uint8)
    ours = quant.e4m3_decode(codes)
    lib = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan], lib[~nan])
    # signed zeros too
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(lib[~nan]))


def test_decode_landmarks():
    d = quant.e4m3_decode
    assert d(0x7E) == 448.0 and d(0xFE) == -448.0
    assert d(0x01) == 2.0 ** -9
    assert d(0x08) == 2.0 ** -6
    assert d(0x07) == 7 * 2.0 ** -9
    assert d(0x38) == 1.0
    assert d(0x00) == 0.0 and not np.signbit(d(0x00))
    assert d(0x80) == 0.0 and np.signbit(d(0x80))
    # 126 distinct positive finite magnitudes plus zero, strictly increasing with the code
    pos = quant.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)


def test_encode_golden_fixture():
    cases = _golden()
    assert len(cases) >= 20
    y = np.array([c[0] for c in cases], dtype=np.float32)
    want = np.array([c[1] for c in cases], dtype=np.uint8)
    got = quant.e4m3_encode(y)
    bad = [(float(y[i]), hex(want[i]), hex(got[i])) for i in range(len(y)) if want[i] != got[i]]
    assert not bad, bad


def test_encode_decode_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = quant.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(quant.e4m3_encode(vals), codes)


def _midpoints():
    pos = quant.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    return (pos[:-1] + pos[1:]) / 2.0


def test_encode_matches_torch_cast_in_range():
    """torch's float32 -> float8_e4m3fn cast is round-to-nearest-even; below 464 it cannot
    overflow, so it must agree with the oracle exactly, signed zero included."""
    rng = np.random.default_rng(123)
    mids = _midpoints().astype(np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    dense = rng.uniform(-460, 460, size=200000).astype(np.float32)
    small = (rng.standard_normal(200000) * 0.01).astype(np.float32)
    logu = np.exp2(rng.uniform(-14, 8.7, size=200000)).astype(np.float32) * rng.choice([-1, 1], 200000)
    y = np.concatenate([near, -near, dense, small, logu.astype(np.float32), np.float32([0.0, -0.0])])
    y = y[np.abs(y) < 464]
    lib = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = quant.e4m3_encode(y)
    mism = np.nonzero(lib != ours)[0]
    assert mism.size == 0, [(float(y[i]), hex(lib[i]), hex(ours[i])) for i in mism[:10]]


def test_encode_saturates():
    y = np.float32([448.0, 448.5, 463.9, 464.0, 470.0, 480.0, 1e30, -448.5, -1e30])
    got = quant.e4m3_encode(y)
    assert got.tolist() == [0x7E] * 6 + [0x7E, 0xFE, 0xFE]


def test_encode_error_bound_half_ulp():
    rng = np.random.default_rng(7)
    y = (rng.standard_normal(100000) * 50).astype(np.float32)
    y = y[np.abs(y) <= 448]
    rec = quant.e4m3_decode(quant.e4m3_encode(y))
    a = np.abs(y.astype(np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    ulp = 2.0 ** (e - 3)  # normals: 3 mantissa bits; subnormal range: 2^-9
    assert np.all(np.abs(rec - y) <= ulp / 2 + 1e-300)


def test_calibrated_scale_amax_over_448():
    from gen import f32_to_bf16_bits
    x = np.float32([[0.5, -3.5, 1.0], [2.0, 0.25, -1.0]])
    bits = f32_to_bf16_bits(x)
    s = quant.e4m3_calibrated_scale(bits)
    assert s == np.float32(3.5) / np.float32(448)
    # the max-envelope value then maps exactly onto the largest finite code
    assert quant.e4m3_quantize(np.float32([-3.5, 3.5]), s).tolist() == [0xFE, 0x7E]


@pytest.mark.parametrize("bug", ["no_tie_even", "truncate", "drop_sign"])
def test_planted_encoder_mistakes_are_caught(bug, monkeypatch):
    """Plant a mistake in a copy of the encoder and check the golden fixture rejects it."""
    pos = quant.e4m3_decode(np.arange(0x7F, dtype=np.uint8))

    def buggy(y):
        y = np.asarray(y, dtype=np.float32)
        a = np.abs(y).astype(np.float64)
        i = np.clip(np.searchsorted(pos, a, side="right") - 1, 0, 0x7E)
        lo, hi = pos[i], pos[np.minimum(i + 1, 0x7E)]
        if bug == "no_tie_even":
            up = (i < 0x7E) & (hi - a <= a - lo)
        elif bug == "truncate":
            up = np.zeros_like(i, dtype=bool)
        else:
            up = (i < 0x7E) & ((hi - a < a - lo) | ((hi - a == a - lo) & (i % 2 == 1)))
        code = np.where(a >= 448, 0x7E, np.where(up, i + 1, i))
        sign = 0 if bug == "drop_sign" else (np.signbit(y).astype(np.int64) << 7)
        return (code | sign).astype(np.uint8)

    cases = _golden()
    y = np.array([c[0] for c in cases], dtype=np.float32)
    want = np.array([c[1] for c in cases], dtype=np.uint8)
    assert not np.array_equal(buggy(y), want)

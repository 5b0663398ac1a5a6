"""Pins for the oracle's int8 per-(token, head) quantiser and slot-pool layouts (CPU only).

Sources: "int8 per-(token,head) KV cache for the Qwen3.8-Flash-Next QSA path" §The finding
worth upstreaming (one scale per (token, head); 256 B of data + 4 B scale = a 260 B inline
record; a side tensor gives the same memory cost) and "SuperPUPS/Qwen3.8-Flash-Next-INT8KV"
§What it buys you (520 bytes per token per GPU for int8 K+V against 1024 for bf16).
"""

import os
from fractions import Fraction

import numpy as np
import pytest

from gen import f32_to_bf16_bits, small_random
from oracle import quant

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "int8_quantize.txt")
D = 256


def _golden():
    cases = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            name, entries, scale, codes = [p.strip() for p in line.split("|")]
            x = np.zeros(D, dtype=np.float32)
            idx = []
            for e in entries.split():
                i, v = e.split(":")
                x[int(i)] = float(v)
                idx.append(int(i))
            want = np.zeros(D, dtype=np.int8)
            for i, c in zip(idx, codes.split()):
                want[i] = int(c)
            cases.append((name, x, np.float32(float(scale)), want))
    return cases


@pytest.mark.parametrize("case", _golden(), ids=lambda c: c[0])
def test_golden_worked_examples(case):
    name, x, scale, want = case
    # the fixture values are exact in bf16, so the bf16 round trip is the identity
    xb = quant.bf16_bits_to_f32(f32_to_bf16_bits(x))
    assert np.array_equal(xb, x)
    codes, s = quant.int8_quantize(xb[None])
    assert s[0] == scale
    assert np.array_equal(codes[0], want)


# ---- exact rational model of the fp32 arithmetic (independent of numpy's float32 ops)

def _round_f32(v: Fraction) -> Fraction:
    """Round a rational to the nearest binary32 value, ties to even (normal range)."""
    if v == 0:
        return Fraction(0)
    sgn = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = Fraction(2) ** (e - 23)
    n = a / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sgn * fl * q


def _round_half_even(v: Fraction) -> int:
    fl = v.numerator // v.denominator
    rem = v - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return fl


def test_matches_exact_rational_model():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((6, D)).astype(np.float32) * np.float32([1, 3, 0.01, 20, 1e-3, 7])[:, None]
    x = quant.bf16_bits_to_f32(f32_to_bf16_bits(x))
    codes, scale = quant.int8_quantize(x)
    for t in range(x.shape[0]):
        amax = max(abs(Fraction(float(v))) for v in x[t])
        s = _round_f32(amax / 127)
        assert Fraction(float(scale[t])) == s
        for d in range(D):
            y = _round_f32(Fraction(float(x[t, d])) / s)
            c = max(-127, min(127, _round_half_even(y)))
            assert codes[t, d] == c, (t, d)


def test_reconstruction_error_at_most_half_scale():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((512, D)).astype(np.float32) * np.exp2(rng.uniform(-8, 8, (512, 1))).astype(np.float32)
    x = quant.bf16_bits_to_f32(f32_to_bf16_bits(x))
    codes, scale = quant.int8_quantize(x)
    err = np.abs(x.astype(np.float64) - codes.astype(np.float64) * scale[:, None].astype(np.float64))
    # scale/2 from rounding to an integer, plus the fp32 quotient's own rounding (2^-24
    # relative): a quotient just below n + 1/2 can round to exactly n + 1/2, then tie away.
    bound = scale[:, None].astype(np.float64) / 2 + np.abs(x.astype(np.float64)) * 2.0 ** -24
    assert np.all(err <= bound)
    assert np.max(err / scale[:, None].astype(np.float64)) > 0.49
    assert np.all(np.max(np.abs(codes.astype(np.int32)), axis=1) == 127)


def test_all_zero_head_gives_zero_scale_and_codes():
    codes, scale = quant.int8_quantize(np.zeros((2, D), dtype=np.float32))
    assert np.all(scale == 0) and np.all(codes == 0)


def test_layout_sizes_and_inline_record():
    wl = small_random(3, num_slots=64, rows=1, topk=4, num_tokens=40)
    kc, vc, ks, vs = quant.write_int8(wl.k_tokens, wl.v_tokens, wl.slot_mapping, 64, "side")
    kr, vr = quant.write_int8(wl.k_tokens, wl.v_tokens, wl.slot_mapping, 64, "inline")
    # 260-byte inline record for head_dim 256; same bytes as codes + side scale
    assert kr.shape[-1] == 260
    assert kc.nbytes + ks.nbytes == kr.nbytes  # identical memory cost
    # K+V bytes per token per head: 520 for int8 against 1024 for bf16
    assert (kr.shape[-1] + vr.shape[-1]) == 520 and 2 * 2 * D == 1024
    assert np.array_equal(kr[..., :D].view(np.int8), kc)
    assert np.array_equal(kr[..., D:].copy().view("<f4")[..., 0], ks)
    raw = kr[wl.slot_mapping[0], 0, D:].tobytes()
    assert raw == ks[wl.slot_mapping[0], 0].astype("<f4").tobytes()


def test_slot_mapping_minus_one_skips_token():
    wl = small_random(4, num_slots=32, rows=1, topk=4, num_tokens=8)
    sm = wl.slot_mapping.copy()
    sm[3] = -1
    kc, vc, ks, vs = quant.write_int8(wl.k_tokens, wl.v_tokens, sm, 32, "side")
    written = set(sm[sm >= 0].tolist())
    for s in range(32):
        if s not in written:
            assert np.all(kc[s] == 0) and ks[s, 0] == 0
    assert wl.slot_mapping[3] not in written


def test_planted_reciprocal_multiply_is_caught():
    """x * (127 / amax) instead of x / (amax / 127) must fail the exact model somewhere."""
    rng = np.random.default_rng(9)
    x = quant.bf16_bits_to_f32(f32_to_bf16_bits(rng.standard_normal((256, D)).astype(np.float32)))
    codes, scale = quant.int8_quantize(x)
    amax = np.max(np.abs(x), axis=1)
    inv = (np.float32(127) / amax).astype(np.float32)
    bad = np.clip(np.rint(x * inv[:, None]), -127, 127).astype(np.int8)
    assert not np.array_equal(bad, codes)

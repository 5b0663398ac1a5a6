"""Pins of the oracle's FP16-activation paths (CPU only).

"[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache" §Purpose: the first validated contract
runs FP16 activations, so q and the new K/V tokens can be IEEE half. The quantisers and the
attention are the same; what changes is the exact widening of the 16-bit inputs, the fp16
pool (the unquantised baseline cache of that contract) and the calibration bins' values.

The widening is pinned against the binary16 definition written out by hand; the int8 and
E4M3 quantisers against the exact rational model and the error bounds on fp16 data; the
attention against torch's float64 dense attention; the calibration statistics against a
hand-worked fp16 fixture.
"""

import math
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from gen import f32_to_f16_bits, small_random
from oracle import attention as att
from oracle import quant
from oracle.calibration import calibration_stats

D = 256


def _binary16_value(b: int) -> float:
    sign = -1.0 if b >> 15 else 1.0
    e = (b >> 10) & 0x1F
    m = b & 0x3FF
    if e == 0x1F:
        return sign * math.inf if m == 0 else math.nan
    if e == 0:
        return sign * m / 1024.0 * 2.0 ** -14
    return sign * (1.0 + m / 1024.0) * 2.0 ** (e - 15)


def test_widening_every_half_against_the_definition():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = quant.act_bits_to_f32(bits, "f16").astype(np.float64)
    ref = np.array([_binary16_value(int(b)) for b in range(1 << 16)])
    assert np.array_equal(got, ref, equal_nan=True)
    num = ~np.isnan(ref)
    assert np.array_equal(np.signbit(got[num]), np.signbit(ref[num]))  # -0 stays -0


def _round_f32(v: Fraction) -> Fraction:
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


def test_int8_on_fp16_tokens_matches_exact_rational_model():
    rng = np.random.default_rng(21)
    x32 = rng.standard_normal((4, D)).astype(np.float32) * np.float32([1, 30, 1e-3, 300])[:, None]
    bits = f32_to_f16_bits(x32)
    x = quant.act_bits_to_f32(bits, "f16")
    codes, scale = quant.int8_quantize(x)
    for t in range(4):
        amax = max(abs(Fraction(float(v))) for v in x[t])
        s = _round_f32(amax / 127)
        assert Fraction(float(scale[t])) == s
        for d in range(0, D, 7):
            y = _round_f32(Fraction(float(x[t, d])) / s)
            fl = y.numerator // y.denominator
            rem = y - fl
            if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
                fl += 1
            assert codes[t, d] == max(-127, min(127, fl)), (t, d)


def test_int8_and_e4m3_writes_of_fp16_tokens_keep_their_error_bounds():
    wl = small_random(22, num_slots=300, rows=1, topk=4, act_dtype="f16", outlier_frac=0.05)
    x = quant.act_bits_to_f32(wl.k_tokens, "f16").astype(np.float64)
    kc, _, ks, _ = quant.write_int8(wl.k_tokens, wl.v_tokens, wl.slot_mapping, 300, "side", dtype="f16")
    sm = wl.slot_mapping
    rec = kc[sm].astype(np.float64) * ks[sm].astype(np.float64)[..., None]
    bound = ks[sm].astype(np.float64)[..., None] / 2 + np.abs(x) * 2.0 ** -24
    assert np.all(np.abs(x - rec) <= bound)
    # E4M3 with the calibrated per-layer scale: half an E4M3 step of the scaled value, times scale
    s = quant.e4m3_calibrated_scale(wl.k_tokens, dtype="f16")
    assert s == np.float32(np.float32(np.max(np.abs(x))) / np.float32(448.0))
    ec, _ = quant.write_e4m3(wl.k_tokens, wl.v_tokens, sm, 300, s, s, dtype="f16")
    y = np.abs(x / np.float64(s))
    step = np.where(y >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(y, 2.0 ** -6))) - 3), 2.0 ** -9)
    err = np.abs(quant.e4m3_decode(ec[sm]) - x / np.float64(s))
    assert np.all(err <= step / 2 * (1 + 2.0 ** -20) + y * 2.0 ** -23)


def test_fp16_attention_equals_dense_attention():
    wl = small_random(23, num_slots=200, rows=3, topk=200, num_tokens=200, act_dtype="f16")
    K = att.f16_pool_fp64(wl.k_tokens[np.argsort(wl.slot_mapping)])
    V = att.f16_pool_fp64(wl.v_tokens[np.argsort(wl.slot_mapping)])
    o, lse = att.gather_attention(wl.q, K, V, wl.topk, wl.softmax_scale, q_dtype="f16")
    q64 = quant.act_bits_to_f32(wl.q, "f16").astype(np.float64)
    for r in range(3):
        k = torch.from_numpy(np.repeat(K.transpose(1, 0, 2), 16, axis=0))
        v = torch.from_numpy(np.repeat(V.transpose(1, 0, 2), 16, axis=0))
        qq = torch.from_numpy(q64[r])[:, None, :]
        ref = F.scaled_dot_product_attention(qq, k, v, scale=wl.softmax_scale)[:, 0, :].numpy()
        lref = torch.logsumexp((qq @ k.transpose(1, 2))[:, 0, :] * wl.softmax_scale, dim=1).numpy()
        assert np.max(np.abs(o[r] - ref)) < 1e-12
        assert np.max(np.abs(lse[r] - lref)) < 1e-12


def test_fp16_calibration_fixture():
    # 0, -0, 1, 2^-24 (smallest fp16 subnormal), 3 * 2^-8, 65504 (largest finite), -464, +inf, nan
    b = np.array([0x0000, 0x8000, 0x3C00, 0x0001, 0x2200, 0x7BFF, 0xDF40, 0x7C00, 0x7E00], dtype=np.uint16)
    st = calibration_stats(b, scale=1.0, dtype="f16")
    assert st["count"] == 7 and st["zeros"] == 2 and st["nonfinite"] == 2
    assert st["amax"] == np.float32(65504.0)
    assert st["below_subnormal"] == 1 and st["subnormal"] == 1 and st["saturated"] == 1
    st = calibration_stats(b, dtype="f16")
    assert st["scale"] == np.float32(np.float32(65504.0) / np.float32(448.0)) and st["saturated"] == 0
    # the same bit patterns read as bf16 are different numbers: the dtype matters
    assert calibration_stats(b, scale=1.0)["amax"] != st["amax"]

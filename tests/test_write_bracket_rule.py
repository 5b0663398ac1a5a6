"""The int8 write's bracket rule, checked on the CPU against IEEE division.

The write kernel forms a code without dividing: with r = fl(1 / scale) it rounds the exact
products x fl(r (1 - 2^-20)) and x fl(r (1 + 2^-20)) to integers (ties to even; on the device one
fused multiply-add with 1.5 2^23 each) and, where the two agree, takes that integer as the code
of the IEEE quotient fl(x / scale); elsewhere it divides. This test emulates those steps exactly
-- fp32 reciprocal and products rounded to nearest, the exact product of two floats in float64
(48 bits fit in 53), numpy's rint -- and checks the rule against numpy's IEEE fp32 division for
every bf16 magnitude up to each of a sweep of absmax values, both signs: agreement always
means the division's code, and the division is rarely needed. ("int8 per-(token,head) KV
cache for the Qwen3.8-Flash-Next QSA path" §The finding worth upstreaming: scale = absmax / 127,
codes rint(x / scale).)
"""

import numpy as np

BRACKET = np.float32(2.0 ** -20)


def _codes(mags_bits, amax_bits):
    x = (mags_bits.astype(np.uint32) << 16).view(np.float32)
    x = np.concatenate([x, -x])
    a = (np.array([amax_bits], dtype=np.uint32) << 16).view(np.float32)[0]
    s = np.float32(a / np.float32(127.0))                  # scale, fp32 IEEE division
    exact = np.rint(x / s)                                 # the code of fl(x / s), ties to even
    r = np.float32(np.float32(1.0) / s)                    # __frcp_rn
    rlo = np.float32(r * np.float32(1.0 - BRACKET))        # fp32 products, rounded to nearest
    rhi = np.float32(r * np.float32(1.0 + BRACKET))
    lo = np.rint(x.astype(np.float64) * np.float64(rlo))   # the exact product, rounded to an integer
    hi = np.rint(x.astype(np.float64) * np.float64(rhi))
    return exact, lo, hi


def test_agreeing_brackets_give_the_division_code():
    rng = np.random.default_rng(4242)
    # absmax bf16 bit patterns: powers of two, their neighbours, and random magnitudes of the
    # range the kernel decides this way (scales in [2^-100, 2^100])
    amaxes = [0x3F80, 0x3F81, 0x3F7F, 0x4000, 0x42FE, 0x4300, 0x3C00, 0x3E4D, 0x4B7F]
    amaxes += [int(b) for b in rng.integers(0x1000, 0x6F00, 40)]
    fallbacks = total = 0
    for ab in amaxes:
        mags = np.arange(0, ab + 1, dtype=np.uint32).astype(np.uint16)
        exact, lo, hi = _codes(mags, ab)
        agree = lo == hi
        assert np.array_equal(lo[agree], exact[agree]), hex(ab)
        assert np.all(np.abs(exact) <= 127)
        fallbacks += int((~agree).sum())
        total += agree.size
    assert fallbacks / total < 1e-3, (fallbacks, total)


def test_exact_ties_always_fall_back():
    """An exact half-integer quotient (here scale = 1: amax = 127) never takes the bracket:
    the two products straddle it, so the division (ties to even) decides."""
    ab = int((np.array([127.0], dtype=np.float32).view(np.uint32)[0] >> 16))
    halves = np.arange(0.5, 127.0, 1.0, dtype=np.float32)
    bits = (halves.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), halves)  # all exact in bf16
    exact, lo, hi = _codes(bits, ab)
    assert np.all(lo != hi)
    assert np.all(exact % 2 == 0)

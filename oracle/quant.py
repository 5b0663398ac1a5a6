"""Oracle quantisers and slot-pool writes (test infrastructure; see the package docstring).

int8 per-(token, head)                [INT8-PR §The finding worth upstreaming; INT8-KV title]
    For one token's head vector x (bf16 widened to fp32, exactly):
        amax  = max_d |x_d|                       (fp32, exact)
        scale = amax / 127                        (fp32 IEEE division)
        c_d   = clamp(rint(x_d / scale), -127, 127)   (fp32 IEEE division, ties to even)
    amax = 0 stores scale 0 and all-zero codes (the pages are silent; reading taken so that
    dequantisation gives 0 instead of 0/0).
    Stored layouts:
        side   : codes [S, Hkv, D] int8 and scales [S, Hkv] fp32 in a separate tensor
        inline : one record of D + 4 bytes per (slot, head): D code bytes then the fp32
                 scale, little-endian (260 B for D = 256, as the page describes)

FP8 E4M3 ("e4m3fn")                    [SCALES §Calibration; E4M3-PR §Why calibrated scale]
    stored        = e4m3fn(x / scale)
    reconstructed = stored * scale
    scale         = observed max envelope / 448
    Encoding: sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0 holds
    the subnormals m/8 * 2^-6 (smallest 2^-9); 0x7F / 0xFF are NaN; 448 is the largest
    finite magnitude. The encoder rounds the fp32 quotient to the nearest representable
    value, ties to the even mantissa, saturates magnitudes above 448 to 448 (the pages
    report saturation as an observable count, i.e. a clamp), and keeps the sign bit, so a
    negative value that rounds to zero is stored as 0x80.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
INT8_QMAX = 127


# --------------------------------------------------------------------------- bf16 widening

def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32. Exact: bf16 is the top half of fp32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen IEEE half bit patterns (uint16) to float32. Exact: every half is a float32."""
    return np.ascontiguousarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def act_bits_to_f32(bits: np.ndarray, dtype: str = "bf16") -> np.ndarray:
    """Widen 16-bit activations of the given type ('bf16' or 'f16') to float32, exactly.

    [E4M3-PR §Purpose: the first validated contract runs FP16 activations] -- the same quantisers apply to
    fp16 K/V; only the widening differs.
    """
    if dtype == "bf16":
        return bf16_bits_to_f32(bits)
    if dtype == "f16":
        return f16_bits_to_f32(bits)
    raise ValueError(f"unknown activation type {dtype!r}")


# --------------------------------------------------------------------------- int8

def int8_quantize(x: np.ndarray):
    """Quantise head vectors x[..., D] (float32) to int8 codes with one fp32 scale each.

    Returns (codes int8 [..., D], scale float32 [...]).
    """
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1)
    scale = (amax / np.float32(INT8_QMAX)).astype(np.float32)
    codes = np.zeros(x.shape, dtype=np.int8)
    nz = scale > 0
    if np.any(nz):
        y = x[nz] / scale[nz][..., None]  # float32 / float32: IEEE round-to-nearest
        c = np.clip(np.rint(y), -INT8_QMAX, INT8_QMAX)  # rint: ties to even
        codes[nz] = c.astype(np.int8)
    return codes, scale


def int8_inline_records(codes: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """Pack codes [..., D] and scales [...] into inline records [..., D + 4] of bytes."""
    D = codes.shape[-1]
    rec = np.zeros(codes.shape[:-1] + (D + 4,), dtype=np.uint8)
    rec[..., :D] = codes.view(np.uint8)
    rec[..., D:] = np.ascontiguousarray(scale, dtype="<f4")[..., None].view(np.uint8)
    return rec


def write_int8(k_bits, v_bits, slot_mapping, num_slots: int, layout: str, dtype: str = "bf16"):
    """Quantise the tokens' K and V heads and store them in a fresh, zeroed slot pool.

    k_bits, v_bits: uint16 bf16 (or fp16, dtype='f16') [T, Hkv, D]; slot_mapping: int [T],
    -1 skips the token.
    layout 'side' returns (k_codes, v_codes, k_scale, v_scale) with codes int8 [S, Hkv, D]
    and scales fp32 [S, Hkv]; 'inline' returns (k_records, v_records) uint8 [S, Hkv, D + 4].
    """
    T, H, D = k_bits.shape
    kc, ks = int8_quantize(act_bits_to_f32(k_bits, dtype))
    vc, vs = int8_quantize(act_bits_to_f32(v_bits, dtype))
    sm = np.asarray(slot_mapping, dtype=np.int64)
    take = sm >= 0
    dst = sm[take]
    if layout == "side":
        k_cache = np.zeros((num_slots, H, D), dtype=np.int8)
        v_cache = np.zeros((num_slots, H, D), dtype=np.int8)
        k_scale = np.zeros((num_slots, H), dtype=np.float32)
        v_scale = np.zeros((num_slots, H), dtype=np.float32)
        k_cache[dst] = kc[take]
        v_cache[dst] = vc[take]
        k_scale[dst] = ks[take]
        v_scale[dst] = vs[take]
        return k_cache, v_cache, k_scale, v_scale
    if layout == "inline":
        k_rec = np.zeros((num_slots, H, D + 4), dtype=np.uint8)
        v_rec = np.zeros((num_slots, H, D + 4), dtype=np.uint8)
        k_rec[dst] = int8_inline_records(kc[take], ks[take])
        v_rec[dst] = int8_inline_records(vc[take], vs[take])
        return k_rec, v_rec
    raise ValueError(f"unknown int8 layout {layout!r}")


# --------------------------------------------------------------------------- E4M3

def e4m3_decode_one(code: int) -> float:
    """Value of one E4M3 byte, from the format's definition."""
    sign = -1.0 if (code >> 7) & 1 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_VALUES = np.array([e4m3_decode_one(c) for c in range(256)], dtype=np.float64)
# codes 0x00..0x7E are the non-negative finite values in increasing order
_E4M3_POS = E4M3_VALUES[:0x7F]


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Decode E4M3 bytes to float64 (exact)."""
    return E4M3_VALUES[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(y: np.ndarray) -> np.ndarray:
    """Encode finite float32 values to E4M3 bytes: nearest value, ties to even, saturate at 448.

    The search is over the table of all representable magnitudes, so the rounding is the
    textbook one: pick the closer neighbour; on an exact tie, the one with an even
    mantissa (an even code, since code order follows value order).
    """
    y = np.asarray(y, dtype=np.float32)
    a = np.abs(y).astype(np.float64)
    i = np.searchsorted(_E4M3_POS, a, side="right") - 1  # largest code with value <= a
    i = np.clip(i, 0, 0x7E)
    lo = _E4M3_POS[i]
    hi = _E4M3_POS[np.minimum(i + 1, 0x7E)]
    d_lo = a - lo
    d_hi = hi - a
    up = (i < 0x7E) & ((d_hi < d_lo) | ((d_hi == d_lo) & (i % 2 == 1)))
    code = np.where(up, i + 1, i)
    code = np.where(a >= E4M3_MAX, 0x7E, code)
    sign = np.signbit(y).astype(np.int64) << 7
    return (code | sign).astype(np.uint8)


def e4m3_calibrated_scale(x_bits: np.ndarray, dtype: str = "bf16") -> np.float32:
    """Per-layer, per-tensor scale = amax / 448 in fp32 over 16-bit values (the max envelope)."""
    amax = np.max(np.abs(act_bits_to_f32(x_bits, dtype)))
    return np.float32(np.float32(amax) / np.float32(E4M3_MAX))


def e4m3_quantize(x: np.ndarray, scale) -> np.ndarray:
    """stored = e4m3fn(x / scale), the quotient in fp32 IEEE division."""
    s = np.float32(scale)
    y = np.asarray(x, dtype=np.float32) / s
    return e4m3_encode(y)


def write_e4m3(k_bits, v_bits, slot_mapping, num_slots: int, k_scale, v_scale, dtype: str = "bf16"):
    """Quantise K and V with their per-layer scales into a fresh, zeroed E4M3 slot pool.

    k_bits, v_bits: uint16 bf16 (or fp16, dtype='f16'). Returns (k_cache, v_cache) uint8 [S, Hkv, D].
    """
    T, H, D = k_bits.shape
    kq = e4m3_quantize(act_bits_to_f32(k_bits, dtype), k_scale)
    vq = e4m3_quantize(act_bits_to_f32(v_bits, dtype), v_scale)
    sm = np.asarray(slot_mapping, dtype=np.int64)
    take = sm >= 0
    k_cache = np.zeros((num_slots, H, D), dtype=np.uint8)
    v_cache = np.zeros((num_slots, H, D), dtype=np.uint8)
    k_cache[sm[take]] = kq[take]
    v_cache[sm[take]] = vq[take]
    return k_cache, v_cache


def write_bf16(k_bits, v_bits, slot_mapping, num_slots: int):
    """Unquantised 16-bit pool (bf16, or fp16 bits alike): the tokens' bits copied to their slots."""
    T, H, D = k_bits.shape
    sm = np.asarray(slot_mapping, dtype=np.int64)
    take = sm >= 0
    k_cache = np.zeros((num_slots, H, D), dtype=np.uint16)
    v_cache = np.zeros((num_slots, H, D), dtype=np.uint16)
    k_cache[sm[take]] = k_bits[take]
    v_cache[sm[take]] = v_bits[take]
    return k_cache, v_cache

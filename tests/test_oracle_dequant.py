"""Pins for the oracle's dequantisation of a slot pool (CPU only).

The attention pins build K and V with these same functions on both sides, so they cannot see
a mistake in the dequantisation itself. These pins compare it with things it does not
compute:

* a hand-worked fixture of stored codes and scales (tests/golden/dequant.txt);
* the original tokens: for every written token t and head h, the value read back from its
  slot must lie within the format's own rounding bound of x[t, h]
  - int8 per-(token, head): |c * scale - x| <= scale / 2 + 2^-24 |x|, the scale/2 of the
    quantiser plus the rounding of the fp32 quotient x / scale
    ("int8 per-(token,head) KV cache for the Qwen3.8-Flash-Next QSA path", §The finding
    worth upstreaming: one scale per (token, head));
  - E4M3: |dec(c) * scale - x| <= (half an E4M3 step at |x / scale|) * scale + 2^-24 |x|
    ("Qwen3.8 Flash Next NVFP4 QSA FP8 E4M3 KV Scales", §Calibration: reconstructed =
    stored * scale);
  - 16-bit pools: exact, checked against torch's own bf16 / fp16 widening;
* single-key attention (o = V_j) read against the token, which fixes where the E4M3 V scale
  is applied ("[Perf][SM70][FP8] Hoist QSA E4M3 KV scales", §Changes: once, after the
  accumulation or after the split-K merge).

Two KV heads with magnitudes 64x apart make a scale taken from the wrong head visible.
Planted mistakes (wrong head, scale omitted, scale applied twice, scale read from the wrong
bytes of an inline record, V scale applied both in the pool and after the merge) must fail.
"""

import os

import numpy as np
import pytest
import torch

from gen import f32_to_bf16_bits, f32_to_f16_bits
from oracle import attention as att
from oracle import quant

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dequant.txt")
D = 256
HEAD_GAIN = (0.25, 16.0)  # per-KV-head magnitude of the synthetic tokens


# --------------------------------------------------------------------------- hand-worked fixture

def _golden():
    rows = {"int8": [], "e4m3": [], "bf16": [], "f16": []}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            parts = [p.strip() for p in line.split("|")]
            rows[parts[0]].append(parts[1:])
    return rows


def _entries(text, conv):
    out = {}
    for e in text.split():
        i, v = e.split(":")
        out[int(i)] = conv(v)
    return out


def test_golden_int8_side_and_inline():
    cases = _golden()["int8"]
    codes = np.zeros((2, 2, D), dtype=np.int8)
    scale = np.zeros((2, 2), dtype=np.float32)
    want = np.zeros((2, 2, D), dtype=np.float64)
    for slot, head, sc, cs, ex in cases:
        j, h = int(slot), int(head)
        scale[j, h] = np.float32(float(sc))
        for d, c in _entries(cs, int).items():
            codes[j, h, d] = c
        for d, v in _entries(ex, float).items():
            want[j, h, d] = v
    got = att.int8_side_pool_fp64(codes, scale)
    assert got.dtype == np.float64 and np.array_equal(got, want)
    # the same records in the inline layout: D code bytes, then the scale's 4 bytes (LE fp32)
    rec = np.zeros((2, 2, D + 4), dtype=np.uint8)
    rec[..., :D] = codes.view(np.uint8)
    for j in range(2):
        for h in range(2):
            rec[j, h, D:] = np.frombuffer(np.float32(scale[j, h]).tobytes(), dtype=np.uint8)
    assert np.array_equal(att.int8_inline_pool_fp64(rec), want)


def test_golden_e4m3_with_and_without_the_scale():
    tensors = {"K": np.float32(0.25), "V": np.float32(2.0)}
    for name, s in tensors.items():
        codes = np.zeros((2, 2, D), dtype=np.uint8)
        want = np.zeros((2, 2, D), dtype=np.float64)
        for slot, head, t, cs, ex in _golden()["e4m3"]:
            if t != name:
                continue
            j, h = int(slot), int(head)
            for d, c in _entries(cs, lambda v: int(v, 16)).items():
                codes[j, h, d] = c
            for d, v in _entries(ex, float).items():
                want[j, h, d] = v
        got = att.e4m3_pool_fp64(codes, s)
        assert np.array_equal(got, want)
        assert np.array_equal(np.signbit(got), np.signbit(want))  # 0x80 reads as -0
        # without the scale: the decoded values alone (the scales are powers of two: exact)
        assert np.array_equal(att.e4m3_pool_fp64(codes, s, apply_scale=False), want / float(s))


def test_golden_16bit_pools():
    for kind, fn in (("bf16", att.bf16_pool_fp64), ("f16", att.f16_pool_fp64)):
        cases = _golden()[kind]
        bits = np.array([int(b, 16) for b, _ in cases], dtype=np.uint16)
        want = np.array([float(v) for _, v in cases], dtype=np.float64)
        got = fn(bits)
        assert np.array_equal(got, want), kind
        assert np.array_equal(np.signbit(got), np.signbit(want)), kind


# --------------------------------------------------------------------------- against the tokens

def _tokens(seed, T=96, H=2, dtype="bf16"):
    """Seeded bf16 (or fp16) tokens [T, H, D], head h scaled by HEAD_GAIN[h], a few outliers."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H, D), dtype=np.float32)
    x *= np.asarray(HEAD_GAIN[:H], dtype=np.float32)[None, :, None]
    x[::17] *= np.float32(12.0)
    to16 = f32_to_f16_bits if dtype == "f16" else f32_to_bf16_bits
    return to16(x)


def _torch_widen(bits, dtype):
    """Token values through torch's own 16-bit widening (a library routine, not the oracle's)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16).to(torch.float64).numpy()


def _written(T, S, seed):
    rng = np.random.default_rng(seed)
    sm = rng.choice(S, size=T, replace=False).astype(np.int64)
    sm[5] = -1  # a skipped token
    return sm


def _check_int8(pool_fn, seed=0, dtype="bf16"):
    """max over written (t, h, d) of |pool - x| / bound; <= 1 passes."""
    k = _tokens(seed, dtype=dtype)
    T, H, _ = k.shape
    S = 160
    sm = _written(T, S, seed + 1)
    x = _torch_widen(k, dtype)
    kc, _, ks, _ = quant.write_int8(k, k, sm, S, "side", dtype=dtype)
    kr, _ = quant.write_int8(k, k, sm, S, "inline", dtype=dtype)
    pool = pool_fn(kc, ks, kr)
    amax = np.max(np.abs(x), axis=-1, keepdims=True)  # [T, H, 1]
    bound = amax / 127.0 / 2.0 * (1 + 2.0 ** -22) + 2.0 ** -24 * np.abs(x)
    take = sm >= 0
    err = np.abs(pool[sm[take]] - x[take])
    return float(np.max(err / bound[take]))


def _side(kc, ks, kr):
    return att.int8_side_pool_fp64(kc, ks)


def _inline(kc, ks, kr):
    return att.int8_inline_pool_fp64(kr)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("fn", [_side, _inline], ids=["side", "inline"])
def test_int8_pool_reads_back_each_token_within_half_a_scale(fn, dtype):
    assert _check_int8(fn, seed=3, dtype=dtype) <= 1.0


def _e4m3_half_step(y):
    """Half the E4M3 grid spacing at |y| (normals: 2^(floor(log2|y|) - 3); below 2^-6: 2^-9)."""
    a = np.abs(y)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    return 0.5 * 2.0 ** (np.minimum(e, 8) - 3)


def _check_e4m3(pool_fn, seed=0, dtype="bf16"):
    k = _tokens(seed, dtype=dtype)
    T, H, _ = k.shape
    S = 160
    sm = _written(T, S, seed + 1)
    x = _torch_widen(k, dtype)
    # per-tensor scale chosen by the test (not by the calibration under test elsewhere): the
    # largest magnitude lands at 400, inside the grid
    s = np.float32(np.max(np.abs(x)) / 400.0)
    kc, _ = quant.write_e4m3(k, k, sm, S, s, s, dtype=dtype)
    pool = pool_fn(kc, s)
    take = sm >= 0
    xt = x[take]
    bound = _e4m3_half_step(xt / float(s)) * float(s) + 2.0 ** -24 * np.abs(xt)
    err = np.abs(pool[sm[take]] - xt)
    return float(np.max(err / bound))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_e4m3_pool_reads_back_each_token_within_half_a_step(dtype):
    assert _check_e4m3(lambda c, s: att.e4m3_pool_fp64(c, s), seed=4, dtype=dtype) <= 1.0
    # without the scale the pool holds x / scale, within half a step of the grid
    unscaled = lambda c, s: att.e4m3_pool_fp64(c, s, apply_scale=False) * float(s)
    assert _check_e4m3(unscaled, seed=4, dtype=dtype) <= 1.0


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_16bit_pools_read_back_each_token_exactly(dtype):
    k = _tokens(5, dtype=dtype)
    sm = _written(k.shape[0], 160, 6)
    kc, _ = quant.write_bf16(k, k, sm, 160)
    pool = att.bf16_pool_fp64(kc) if dtype == "bf16" else att.f16_pool_fp64(kc)
    take = sm >= 0
    assert np.array_equal(pool[sm[take]], _torch_widen(k, dtype)[take])
    assert np.all(pool[np.setdiff1d(np.arange(160), sm[take])] == 0)


# --------------------------------------------------------------------------- planted mistakes

def _side_wrong_head(kc, ks, kr):
    return kc.astype(np.float64) * ks.astype(np.float64)[:, ::-1, None]


def _side_no_scale(kc, ks, kr):
    return kc.astype(np.float64)


def _side_scale_twice(kc, ks, kr):
    s = ks.astype(np.float64)[..., None]
    return kc.astype(np.float64) * s * s


def _inline_scale_from_wrong_bytes(kr, kc=None, ks=None):
    codes = np.ascontiguousarray(kr[..., :D]).view(np.int8)
    scale = np.ascontiguousarray(kr[..., D - 4:D]).view("<f4")[..., 0]  # the last code bytes
    return codes.astype(np.float64) * np.nan_to_num(scale.astype(np.float64))[..., None]


def _inline_scale_big_endian(kr, kc=None, ks=None):
    codes = np.ascontiguousarray(kr[..., :D]).view(np.int8)
    scale = np.ascontiguousarray(kr[..., D:]).view(">f4")[..., 0]
    return codes.astype(np.float64) * np.nan_to_num(scale.astype(np.float64), posinf=0, neginf=0)[..., None]


@pytest.mark.parametrize("bad", [_side_wrong_head, _side_no_scale, _side_scale_twice])
def test_planted_int8_side_mistakes_fail_the_token_pin(bad):
    assert _check_int8(bad, seed=3) > 1.0


@pytest.mark.parametrize("bad", [_inline_scale_from_wrong_bytes, _inline_scale_big_endian])
def test_planted_int8_inline_mistakes_fail_the_token_pin(bad):
    assert _check_int8(lambda kc, ks, kr: bad(kr), seed=3) > 1.0


@pytest.mark.parametrize("bad", [
    lambda c, s: quant.e4m3_decode(c),                                   # scale omitted
    lambda c, s: quant.e4m3_decode(c) * float(s) * float(s),            # applied twice
    lambda c, s: quant.e4m3_decode(c ^ np.uint8(0x80)) * float(s),      # sign bit flipped
    lambda c, s: quant.e4m3_decode(c) * float(s) * 2.0,                 # exponent bias off by one
])
def test_planted_e4m3_mistakes_fail_the_token_pin(bad):
    assert _check_e4m3(bad, seed=4) > 1.0


def test_planted_16bit_mistake_fails():
    k = _tokens(5)
    wrong = (np.asarray(k, dtype=np.uint32) << np.uint32(15)).view(np.float32).astype(np.float64)
    assert not np.array_equal(wrong, _torch_widen(k, "bf16"))
    assert np.array_equal(att.bf16_pool_fp64(k), _torch_widen(k, "bf16"))


# --------------------------------------------------------------------------- single-key attention

def _single_key_rows(S, sm, n_rows, seed):
    rng = np.random.default_rng(seed)
    written = sm[sm >= 0]
    idx = np.full((n_rows, 3), -1, dtype=np.int32)
    idx[:, 1] = rng.choice(written, size=n_rows, replace=False)  # one valid key among padding
    return idx


def _v_token_for(idx, sm, v):
    inv = {int(s): t for t, s in enumerate(sm) if s >= 0}
    return np.stack([v[inv[int(j)]] for j in idx[:, 1]])  # [R, H, D]


def test_single_key_attention_returns_the_tokens_value_row_for_each_format():
    """k = 1 valid key: o[r, g] = V of that key's KV head, read back against the token itself."""
    T, H, G, R = 96, 2, 3, 8
    kb, vb = _tokens(7), _tokens(8)
    sm = _written(T, 160, 9)
    q = f32_to_bf16_bits(np.random.default_rng(10).standard_normal((R, H * G, D), dtype=np.float32))
    idx = _single_key_rows(160, sm, R, 11)
    v = _torch_widen(vb, "bf16")
    vt = _v_token_for(idx, sm, v)  # [R, H, D]
    vt_g = np.repeat(vt, G, axis=1)  # query head g reads KV head g // G

    kc, vc, ks, vs = quant.write_int8(kb, vb, sm, 160, "side")
    o, _ = att.gather_attention(q, att.int8_side_pool_fp64(kc, ks), att.int8_side_pool_fp64(vc, vs), idx, 1 / 16)
    amax = np.repeat(np.max(np.abs(vt), axis=-1, keepdims=True), G, axis=1)
    assert np.all(np.abs(o - vt_g) <= amax / 254.0 * (1 + 2.0 ** -22) + 2.0 ** -24 * np.abs(vt_g))

    s_k = np.float32(np.max(np.abs(_torch_widen(kb, "bf16"))) / 400.0)
    s_v = np.float32(np.max(np.abs(v)) / 400.0)
    kc, vc = quant.write_e4m3(kb, vb, sm, 160, s_k, s_v)
    Kd = att.e4m3_pool_fp64(kc, s_k, apply_scale=False)
    Vd = att.e4m3_pool_fp64(vc, s_v, apply_scale=False)
    bound = _e4m3_half_step(vt_g / float(s_v)) * float(s_v) + 2.0 ** -24 * np.abs(vt_g)
    # the hoisted order: partials without the V scale, the scale once after the merge
    op, lp = att.gather_attention_splits(q, Kd, Vd, idx, float(s_k) / 16, 3)
    o, _ = att.merge_splits(op, lp, v_scale_post=float(s_v))
    assert np.all(np.abs(o - vt_g) <= bound)
    # planted: the V scale applied in the pool and again after the merge
    op, lp = att.gather_attention_splits(q, Kd, att.e4m3_pool_fp64(vc, s_v), idx, float(s_k) / 16, 3)
    o_bad, _ = att.merge_splits(op, lp, v_scale_post=float(s_v))
    assert not np.all(np.abs(o_bad - vt_g) <= bound)

    kc, vc = quant.write_bf16(kb, vb, sm, 160)
    o, _ = att.gather_attention(q, att.bf16_pool_fp64(kc), att.bf16_pool_fp64(vc), idx, 1 / 16)
    assert np.array_equal(o, vt_g)

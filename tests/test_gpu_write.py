"""GPU parity of the quantize-on-write kernels: stored bytes and scales must equal the CPU
oracle's bit for bit ("int8 per-(token,head) KV cache for the Qwen3.8-Flash-Next QSA path"
§The finding worth upstreaming; "Qwen3.8 Flash Next NVFP4 QSA FP8 E4M3 KV Scales"
§Calibration)."""

import numpy as np
import pytest
import torch

from gen import chunked_prefill, e4m3_splitk_layer, small_random, tiny
from oracle import quant as oq

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import quantized_kv_cache_write_gb300 as q
    return q


def _cases():
    return {
        "tiny": lambda: tiny(0),
        "ragged_zero_heads": lambda: small_random(31, num_slots=5000, rows=1, topk=1, num_tokens=777,
                                                  num_kv_heads=2, num_q_heads=4, outlier_frac=0.02,
                                                  zero_tokens=5),
        "prefill_8192_into_524288": lambda: chunked_prefill(4),
        "two_heads_9000_tokens": lambda: small_random(41, num_slots=12000, rows=1, topk=1, num_tokens=9000,
                                                      num_kv_heads=2, num_q_heads=4, outlier_frac=0.02,
                                                      zero_tokens=7),
    }


@pytest.mark.parametrize("case", list(_cases()))
@pytest.mark.parametrize("layout", ["int8_side", "int8_inline"])
def test_int8_write_bit_exact(q, case, layout):
    wl = _cases()[case]()
    from harness import GpuPool
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool = GpuPool(wl, layout, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    ref = oq.write_int8(wl.k_tokens, wl.v_tokens, wl.slot_mapping, wl.num_slots,
                        "side" if layout == "int8_side" else "inline")
    if layout == "int8_side":
        got = [pool.k_cache, pool.v_cache, pool.k_scale_tok, pool.v_scale_tok]
    else:
        got = [pool.k_cache, pool.v_cache]
    for g, r in zip(got, ref):
        g = g.cpu().numpy()
        assert g.view(np.uint8).tobytes() == np.ascontiguousarray(r).view(np.uint8).tobytes()


@pytest.mark.parametrize("case", list(_cases()) + ["e4m3_layer"])
def test_e4m3_calibrate_and_write_bit_exact(q, case):
    wl = e4m3_splitk_layer(0) if case == "e4m3_layer" else _cases()[case]()
    from harness import GpuPool
    pool = GpuPool(wl, "e4m3")
    ks = oq.e4m3_calibrated_scale(wl.k_tokens)
    vs = oq.e4m3_calibrated_scale(wl.v_tokens)
    assert np.float32(pool.k_scale_layer).tobytes() == ks.tobytes()
    assert np.float32(pool.v_scale_layer).tobytes() == vs.tobytes()
    kc, vc = oq.write_e4m3(wl.k_tokens, wl.v_tokens, wl.slot_mapping, wl.num_slots, ks, vs)
    assert np.array_equal(pool.k_cache.cpu().numpy(), kc)
    assert np.array_equal(pool.v_cache.cpu().numpy(), vc)


def test_e4m3_write_with_foreign_scale_saturates_and_keeps_signed_zero(q):
    """A scale far below amax/448 forces saturation; a huge one forces underflow to +-0."""
    wl = small_random(32, num_slots=600, rows=1, topk=1, num_tokens=512, zero_tokens=4)
    k = torch.from_numpy(wl.k_tokens.view(np.int16)).view(torch.bfloat16).cuda()
    v = torch.from_numpy(wl.v_tokens.view(np.int16)).view(torch.bfloat16).cuda()
    slots = torch.from_numpy(wl.slot_mapping).cuda()
    for ks, vs in [(np.float32(1e-3), np.float32(3e-3)), (np.float32(1e4), np.float32(1.0))]:
        kc = torch.zeros((600, 1, 256), dtype=torch.uint8, device="cuda")
        vc = torch.zeros_like(kc)
        q.qkv_write_e4m3(k, v, slots, kc, vc, float(ks), float(vs))
        rk, rv = oq.write_e4m3(wl.k_tokens, wl.v_tokens, wl.slot_mapping, 600, ks, vs)
        assert np.array_equal(kc.cpu().numpy(), rk)
        assert np.array_equal(vc.cpu().numpy(), rv)
    assert np.any(rk == 0x80) and np.any(rk == 0x00)


@pytest.mark.parametrize("num_tokens", [200, 20000])  # 20000: each warp writes a head's K and V rows
def test_bad_slots_are_flagged_and_skipped(q, num_tokens):
    S = num_tokens + 100
    wl = small_random(33, num_slots=S, rows=1, topk=1, num_tokens=num_tokens)
    sm = wl.slot_mapping.copy()
    sm[[3, 50]] = [S, -7]  # out of range
    sm[[7, num_tokens - 1]] = -1  # skip
    k = torch.from_numpy(wl.k_tokens.view(np.int16)).view(torch.bfloat16).cuda()
    v = torch.from_numpy(wl.v_tokens.view(np.int16)).view(torch.bfloat16).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kc = torch.full((S, 1, 256), 0x5A, dtype=torch.int8, device="cuda")
    vc = kc.clone()
    ks = torch.full((S, 1), -1.0, dtype=torch.float32, device="cuda")
    vs = ks.clone()
    q.qkv_write_int8(k, v, torch.from_numpy(sm).cuda(), kc, vc, ks, vs, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == q.QKV_DEV_BAD_SLOT
    okm = sm.copy()
    okm[[3, 50]] = -1
    rk, rv, rks, rvs = oq.write_int8(wl.k_tokens, wl.v_tokens, okm, S, "side")
    written = okm[okm >= 0]
    untouched = np.setdiff1d(np.arange(S), written)
    for got, ref in ((kc, rk), (vc, rv), (ks, rks), (vs, rvs)):
        assert np.array_equal(got.cpu().numpy()[written], ref[written])
    assert np.all(kc.cpu().numpy()[untouched] == 0x5A) and np.all(ks.cpu().numpy()[untouched] == -1.0)
    assert np.all(vc.cpu().numpy()[untouched] == 0x5A) and np.all(vs.cpu().numpy()[untouched] == -1.0)


def test_strided_tokens_from_a_fused_kv_buffer(q):
    """K and V as views into one [T, 2, Hkv, D] buffer (token stride 2*Hkv*D)."""
    wl = small_random(34, num_slots=400, rows=1, topk=1, num_tokens=300, num_kv_heads=2, num_q_heads=4)
    fused = np.stack([wl.k_tokens, wl.v_tokens], axis=1)  # [T, 2, H, D]
    fd = torch.from_numpy(np.ascontiguousarray(fused).view(np.int16)).view(torch.bfloat16).cuda()
    k, v = fd[:, 0], fd[:, 1]
    kc = torch.zeros((400, 2, 256), dtype=torch.int8, device="cuda")
    vc = torch.zeros_like(kc)
    ks = torch.zeros((400, 2), dtype=torch.float32, device="cuda")
    vs = torch.zeros_like(ks)
    q.qkv_write_int8(k, v, torch.from_numpy(wl.slot_mapping).cuda(), kc, vc, ks, vs)
    rk, rv, rks, rvs = oq.write_int8(wl.k_tokens, wl.v_tokens, wl.slot_mapping, 400, "side")
    assert np.array_equal(kc.cpu().numpy(), rk) and np.array_equal(vc.cpu().numpy(), rv)
    assert np.array_equal(ks.cpu().numpy(), rks) and np.array_equal(vs.cpu().numpy(), rvs)


def test_empty_write_and_calibrate_of_zeros(q):
    k = torch.zeros((0, 1, 256), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((4, 1, 256), dtype=torch.int8, device="cuda")
    ks = torch.zeros((4, 1), dtype=torch.float32, device="cuda")
    q.qkv_write_int8(k, k, torch.zeros(0, dtype=torch.int64, device="cuda"), kc, kc, ks, ks)
    z = torch.zeros(1000, dtype=torch.bfloat16, device="cuda")
    amax = torch.ones(1, dtype=torch.int32, device="cuda")
    sc = torch.full((1,), 7.0, dtype=torch.float32, device="cuda")
    q.qkv_e4m3_calibrate(z, amax, sc)
    assert sc.item() == 0.0


def _magnitude_sweep_heads(amax_list, seed):
    """Heads of 256 16-bit values: the amax A first, then every magnitude pattern at or below A
    with random signs (zero-padded to whole heads). For one A this is every quotient x / scale a
    head of that scale can form, so rounding ties and near-ties all occur."""
    rng = np.random.default_rng(seed)
    heads = []
    for A in amax_list:
        mags = np.arange(0, A + 1, dtype=np.uint32).astype(np.uint16)
        vals = mags | (rng.integers(0, 2, mags.size).astype(np.uint16) << np.uint16(15))
        vals = np.concatenate([vals, np.zeros((-vals.size) % 255, dtype=np.uint16)]).reshape(-1, 255)
        heads.append(np.concatenate([np.full((vals.shape[0], 1), A, dtype=np.uint16), vals], axis=1))
    return np.concatenate(heads)


def _dev16(bits, dtype):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    return t.view(torch.float16 if dtype == "f16" else torch.bfloat16)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("layout", ["side", "inline"])
@pytest.mark.parametrize("large", [False, True])
def test_int8_write_exhaustive_over_magnitudes(q, dtype, layout, large):
    """Every 16-bit magnitude up to each head's amax, for amaxes from subnormal to the largest
    finite value: stored codes and scales equal the oracle's bit for bit. `large` repeats the
    tokens past 16384 (token, head) units, where each warp writes a head's K and V rows."""
    if dtype == "bf16":
        amax = [0x3F80, 0x3E4D, 0x4300, 0x4B7F, 0x5F00, 0x7F7F, 0x0D00, 0x0200, 0x0050]
    else:
        amax = [0x3C00, 0x2E66, 0x5800, 0x7BFF, 0x0400, 0x0123, 0x0001]
    k = _magnitude_sweep_heads(amax, 1)[:, None, :]
    v = _magnitude_sweep_heads(amax, 2)[:, None, :]
    if large:
        reps = -(-16384 // k.shape[0]) + 1
        k, v = np.tile(k, (reps, 1, 1)), np.tile(v[::-1], (reps, 1, 1))
    T = k.shape[0]
    slots_np = np.random.default_rng(3).permutation(T).astype(np.int64)
    D = 256
    slots = torch.from_numpy(slots_np).cuda()
    if layout == "side":
        kc = torch.zeros((T, 1, D), dtype=torch.int8, device="cuda")
        vc = torch.zeros_like(kc)
        ks = torch.zeros((T, 1), dtype=torch.float32, device="cuda")
        vs = torch.zeros_like(ks)
        q.qkv_write_int8(_dev16(k, dtype), _dev16(v, dtype), slots, kc, vc, ks, vs)
        got = [kc, vc, ks, vs]
    else:
        kc = torch.zeros((T, 1, D + 4), dtype=torch.uint8, device="cuda")
        vc = torch.zeros_like(kc)
        q.qkv_write_int8(_dev16(k, dtype), _dev16(v, dtype), slots, kc, vc, layout=q.QKV_INT8_INLINE)
        got = [kc, vc]
    ref = oq.write_int8(k, v, slots_np, T, layout, dtype=dtype)
    for g, r in zip(got, ref):
        assert g.cpu().numpy().view(np.uint8).tobytes() == np.ascontiguousarray(r).view(np.uint8).tobytes()


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_e4m3_write_exhaustive_over_values(q, dtype):
    """Every finite 16-bit value of both signs, at scales from subnormal to 1e38 (multiply
    path and division path): stored codes equal the oracle's bit for bit."""
    top = 0x7F7F if dtype == "bf16" else 0x7BFF
    mags = np.arange(0, top + 1, dtype=np.uint32).astype(np.uint16)
    vals = np.concatenate([mags, mags | np.uint16(0x8000)])
    vals = np.concatenate([vals, np.zeros((-vals.size) % 256, dtype=np.uint16)]).reshape(-1, 1, 256)
    T = vals.shape[0]
    k, v = vals, vals[::-1].copy()
    slots_np = np.arange(T, dtype=np.int64)
    slots = torch.from_numpy(slots_np).cuda()
    kc = torch.zeros((T, 1, 256), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    for ks, vs in [(0.0173, 1.0), (3.7e-3, 2.0 ** -20), (1e-37, 3e37), (1e-39, 1e38), (448.0, 7.1e-5)]:
        ks32, vs32 = np.float32(ks), np.float32(vs)
        q.qkv_write_e4m3(_dev16(k, dtype), _dev16(v, dtype), slots, kc, vc, float(ks32), float(vs32))
        rk, rv = oq.write_e4m3(k, v, slots_np, T, ks32, vs32, dtype=dtype)
        assert np.array_equal(kc.cpu().numpy(), rk), (ks, vs)
        assert np.array_equal(vc.cpu().numpy(), rv), (ks, vs)

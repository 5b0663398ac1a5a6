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


def test_bad_slots_are_flagged_and_skipped(q):
    wl = small_random(33, num_slots=300, rows=1, topk=1, num_tokens=200)
    sm = wl.slot_mapping.copy()
    sm[[3, 50]] = [300, -7]  # out of range
    sm[7] = -1  # skip
    k = torch.from_numpy(wl.k_tokens.view(np.int16)).view(torch.bfloat16).cuda()
    v = torch.from_numpy(wl.v_tokens.view(np.int16)).view(torch.bfloat16).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kc = torch.full((300, 1, 256), 0x5A, dtype=torch.int8, device="cuda")
    vc = kc.clone()
    ks = torch.full((300, 1), -1.0, dtype=torch.float32, device="cuda")
    vs = ks.clone()
    q.qkv_write_int8(k, v, torch.from_numpy(sm).cuda(), kc, vc, ks, vs, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == q.QKV_DEV_BAD_SLOT
    okm = sm.copy()
    okm[[3, 50]] = -1
    rk, rv, rks, rvs = oq.write_int8(wl.k_tokens, wl.v_tokens, okm, 300, "side")
    written = okm[okm >= 0]
    untouched = np.setdiff1d(np.arange(300), written)
    assert np.array_equal(kc.cpu().numpy()[written], rk[written])
    assert np.array_equal(ks.cpu().numpy()[written], rks[written])
    assert np.all(kc.cpu().numpy()[untouched] == 0x5A) and np.all(ks.cpu().numpy()[untouched] == -1.0)


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

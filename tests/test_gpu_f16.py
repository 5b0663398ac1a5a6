"""FP16-activation paths on the GPU against the oracle.

"[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache" §Purpose: the first validated contract
runs FP16 activations. q and the new K/V tokens are IEEE half: the writes must store the
oracle's bytes exactly, the gather (int8 side / inline, E4M3 and an fp16 pool) must match the
fp64 oracle within |gpu - ref| <= 5e-5 + 1e-3 |ref|, and the calibration statistics of half
tensors must match exactly.
"""

import numpy as np
import pytest
import torch

from gen import small_random
from harness import GpuPool, OraclePool, act_dev, assert_close
from oracle.calibration import calibration_stats

pytestmark = pytest.mark.gpu
FORMATS = ["int8_side", "int8_inline", "e4m3", "f16"]


def _wl(seed, **kw):
    base = dict(num_slots=4000, rows=5, topk=515, pad_frac=0.05, outlier_frac=0.02, act_dtype="f16")
    base.update(kw)
    return small_random(seed, **base)


@pytest.mark.parametrize("fmt", ["int8_side", "int8_inline", "e4m3"])
def test_writes_of_fp16_tokens_are_bit_exact(fmt):
    wl = _wl(81, zero_tokens=3)
    gp, op = GpuPool(wl, fmt), OraclePool(wl, fmt)
    if fmt == "int8_side":
        got = (gp.k_cache, gp.v_cache, gp.k_scale_tok, gp.v_scale_tok)
    else:
        got = (gp.k_cache, gp.v_cache)
    for g, r in zip(got, op.bytes):
        assert g.cpu().numpy().tobytes() == np.ascontiguousarray(r).tobytes()
    if fmt == "e4m3":
        assert np.float32(gp.k_scale_layer) == op.k_scale_layer
        assert np.float32(gp.v_scale_layer) == op.v_scale_layer


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("P", [1, 5])
def test_fp16_query_gather_matches_oracle(fmt, P):
    wl = _wl(82)
    wl.topk[1] = -1  # an empty row
    gp, op = GpuPool(wl, fmt), OraclePool(wl, fmt)
    out, lse, o_part, lse_part = gp.attend(wl, num_splits=P)
    ro, rl = op.attend(wl)
    assert_close(out, ro, f"{fmt} out")
    assert_close(lse, rl, f"{fmt} lse")
    assert np.all(out[1] == 0) and np.all(lse[1] == -np.inf)
    if P > 1:
        po, pl = op.attend_splits(wl, P)
        assert_close(o_part, po, f"{fmt} o_part")
        assert_close(lse_part, pl, f"{fmt} lse_part")


@pytest.mark.parametrize("fmt", ["int8_side", "e4m3", "f16"])
def test_fp16_outlier_heavy_and_gqa32(fmt):
    for seed in range(4):
        wl = _wl(90 + seed, topk=200 + 150 * seed, outlier_frac=0.03 + 0.005 * seed, num_q_heads=32 if seed % 2 else 16)
        out, lse, _, _ = GpuPool(wl, fmt).attend(wl)
        ro, rl = OraclePool(wl, fmt).attend(wl)
        assert_close(out, ro, f"{fmt} out seed {seed}")
        assert_close(lse, rl, f"{fmt} lse seed {seed}")


def test_pool_and_query_types_must_match():
    import quantized_kv_cache_write_gb300 as q
    wl = _wl(83, rows=2, topk=20)
    gp = GpuPool(wl, "f16")
    idx = torch.from_numpy(wl.topk).cuda()
    out = torch.empty((2, 16, 256), dtype=torch.float32, device="cuda")
    qb = act_dev(wl.q, "bf16")  # the same bits read as bf16: wrong type for an fp16 pool
    with pytest.raises(q.QKVError):
        q.qsa_gather_attn(qb, q.QKV_F16, gp.k_cache, gp.v_cache, idx, wl.softmax_scale, out=out)
    with pytest.raises(q.QKVError):
        q.qsa_gather_attn(act_dev(wl.q, "f16"), q.QKV_BF16, gp.k_cache, gp.v_cache, idx, wl.softmax_scale,
                          out=out)


@pytest.mark.parametrize("scale", [0.0, 1.0, 0.05])
def test_fp16_calibration_statistics(scale):
    import quantized_kv_cache_write_gb300 as q
    rng = np.random.default_rng(84)
    x = (rng.standard_normal(200_003) * np.exp2(rng.integers(-20, 8, 200_003))).astype(np.float16)
    x[:5] = [0.0, -0.0, np.inf, 65504.0, 6e-8]
    bits = x.view(np.uint16)
    hist = torch.zeros(q.CALIB_BINS, dtype=torch.int64, device="cuda")
    q.qkv_calib_histogram(act_dev(bits, "f16"), hist)
    rec = torch.zeros(8, dtype=torch.int64, device="cuda")
    q.qkv_calib_stats(hist, rec, scale, dtype=torch.float16)
    got = q.decode_calib_stats(rec)
    ref = calibration_stats(bits, None if scale == 0.0 else scale, dtype="f16")
    for k in ("count", "zeros", "nonfinite", "below_subnormal", "subnormal", "saturated"):
        assert got[k] == ref[k], k
    for k in ("amax", "p99_9", "p99_99", "scale"):
        assert np.float32(got[k]) == np.float32(ref[k]), k

"""Device calibration statistics against the oracle (GPU).

"Qwen3.8 Flash Next NVFP4 QSA FP8 E4M3 KV Scales" §Calibration (max-abs, p99.9, p99.99,
saturation, scale = max / 448) and "[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache"
§Why calibrated scale is part of this contract (elements below 2^-9 and in [2^-9, 2^-6) at a
given scale). Every field is exact (integer counts, or values the input holds), so the GPU
must match the oracle exactly.
"""

import numpy as np
import pytest
import torch

from gen import e4m3_splitk_layer, tiny
from gen.workloads import f32_to_bf16_bits
from oracle.calibration import calibration_stats, magnitude_histogram

pytestmark = pytest.mark.gpu


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).cuda()


def _gpu_stats(chunks, scale=0.0):
    import quantized_kv_cache_write_gb300 as q
    hist = torch.zeros(q.CALIB_BINS, dtype=torch.int64, device="cuda")
    for c in chunks:
        q.qkv_calib_histogram(_dev(c), hist)
    buf = torch.full((8,), -1, dtype=torch.int64, device="cuda")
    q.qkv_calib_stats(hist, buf, scale)
    torch.cuda.synchronize()
    return hist.cpu().numpy(), q.decode_calib_stats(buf)


def _compare(got, ref):
    for k in ("count", "zeros", "nonfinite", "below_subnormal", "subnormal", "saturated"):
        assert got[k] == ref[k], (k, got[k], ref[k])
    for k in ("amax", "p99_9", "p99_99", "scale"):
        assert np.float32(got[k]) == np.float32(ref[k]), (k, got[k], ref[k])


def _mix(seed, n):
    """Normals spread over many octaves, some zeros, tiny values and large outliers."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(n).astype(np.float32) * np.exp2(rng.integers(-14, 4, n)).astype(np.float32)
    x[rng.random(n) < 0.01] = 0.0
    x[rng.random(n) < 0.001] *= np.float32(600.0)
    return f32_to_bf16_bits(x)


@pytest.mark.parametrize("n", [1, 7, 8, 9, 1000, 65537, 3_000_001])
@pytest.mark.parametrize("scale", [0.0, 1.0, 0.0171247218])
def test_histogram_and_stats_match_oracle(n, scale):
    b = _mix(n, n)
    hist, st = _gpu_stats([b], scale)
    assert np.array_equal(hist, magnitude_histogram(b))
    _compare(st, calibration_stats(b, None if scale == 0.0 else scale))


def test_special_values_and_accumulation_over_calls():
    special = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x0001, 0x3F80, 0xC3E8], dtype=np.uint16)
    parts = [_mix(1, 1001), special, _mix(2, 4096), _mix(3, 17)]
    whole = np.concatenate(parts)
    hist, st = _gpu_stats(parts, 1.0)
    assert np.array_equal(hist, magnitude_histogram(whole))
    ref = calibration_stats(whole, 1.0)
    assert ref["nonfinite"] == 3
    _compare(st, ref)


def test_all_zero_tensor():
    _, st = _gpu_stats([np.zeros(100, dtype=np.uint16)])
    assert st["scale"] == 0.0 and st["amax"] == 0.0 and st["zeros"] == 100 and st["count"] == 100
    assert st["below_subnormal"] == st["subnormal"] == st["saturated"] == 0


@pytest.mark.parametrize("tensor", ["k", "v"])
def test_layer_tensor_of_the_split_k_workload(tensor):
    """One layer's K (or V) pool of the E4M3 split-K workload: 131072 x 256 values."""
    wl = e4m3_splitk_layer(0)
    b = (wl.k_tokens if tensor == "k" else wl.v_tokens).ravel()
    for scale in (0.0, 1.0):
        _, st = _gpu_stats([b], scale)
        ref = calibration_stats(b, None if scale == 0.0 else scale)
        _compare(st, ref)
    assert st["saturated"] == 0


def test_calibrated_scale_agrees_with_qkv_e4m3_calibrate():
    import quantized_kv_cache_write_gb300 as q
    wl = tiny(0)
    x = _dev(wl.k_tokens.ravel())
    amax = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc = torch.zeros(1, dtype=torch.float32, device="cuda")
    q.qkv_e4m3_calibrate(x, amax, sc)
    _, st = _gpu_stats([wl.k_tokens.ravel()])
    assert np.float32(st["scale"]) == sc.cpu().numpy()[0]
    assert st["saturated"] == 0

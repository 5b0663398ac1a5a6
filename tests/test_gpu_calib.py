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


def _crafted_histogram(seed, dtype):
    """A sparse histogram with counts on bins at row (32), warp-range (1024) and finite /
    non-finite edges, and the magnitudes it counts, each with a random sign."""
    rng = np.random.default_rng(seed)
    fnf = 0x7F80 if dtype == "bf16" else 0x7C00  # first non-finite magnitude
    edges = np.array([0, 1, 31, 32, 33, 1023, 1024, 1025, 2047, 2048, 16383, 16384, fnf - 1, fnf, fnf + 1, 32767])
    bins = np.unique(np.concatenate([edges[rng.random(edges.size) < 0.7], rng.integers(0, 32768, 40)]))
    counts = rng.integers(1, 2000, bins.size)
    hist = np.zeros(32768, dtype=np.int64)
    hist[bins] = counts
    bits = np.repeat(bins.astype(np.uint16), counts)
    bits |= (rng.integers(0, 2, bits.size).astype(np.uint16) << np.uint16(15))
    return hist, bits


def _bin_f32(b, dtype):
    if dtype == "bf16":
        return np.array([b << 16], dtype=np.uint32).view(np.float32)[0]
    return np.float32(np.array([b], dtype=np.uint16).view(np.float16)[0])


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("seed", range(6))
def test_stats_of_crafted_histograms(dtype, seed):
    """The stats pass alone, fed histograms built on the host: ranks and class edges that fall
    on row and warp-range boundaries, scales that put a bin exactly on 2^-9 or 2^-6 or next
    to 464, and scales that put every element in one class."""
    import quantized_kv_cache_write_gb300 as q
    hist, bits = _crafted_histogram(100 + seed, dtype)
    fnf = 0x7F80 if dtype == "bf16" else 0x7C00
    finite = np.nonzero(hist[1:fnf])[0] + 1
    rng = np.random.default_rng(seed)
    b = int(rng.choice(finite))
    v = _bin_f32(b, dtype)
    scales = [0.0, 1.0, float(v * np.float32(512.0)), float(v * np.float32(64.0)), float(v / np.float32(464.0)),
              1e-30, 1e30]
    hd = torch.from_numpy(hist).cuda()
    buf = torch.full((8,), -1, dtype=torch.int64, device="cuda")
    for scale in scales:
        if not (np.isfinite(scale) and scale >= 0.0):
            continue
        q.qkv_calib_stats(hd, buf, scale, dtype=torch.float16 if dtype == "f16" else torch.bfloat16)
        torch.cuda.synchronize()
        _compare(q.decode_calib_stats(buf), calibration_stats(bits, None if scale == 0.0 else scale, dtype=dtype))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_stats_of_only_non_finite_values(dtype):
    import quantized_kv_cache_write_gb300 as q
    fnf = 0x7F80 if dtype == "bf16" else 0x7C00
    hist = np.zeros(32768, dtype=np.int64)
    hist[[fnf, fnf + 5, 32767]] = [3, 2, 1]
    bits = np.repeat(np.array([fnf, fnf + 5, 32767], dtype=np.uint16), [3, 2, 1])
    buf = torch.full((8,), -1, dtype=torch.int64, device="cuda")
    for scale in (0.0, 2.0):
        q.qkv_calib_stats(torch.from_numpy(hist).cuda(), buf, scale,
                          dtype=torch.float16 if dtype == "f16" else torch.bfloat16)
        got = q.decode_calib_stats(buf)
        _compare(got, calibration_stats(bits, None if scale == 0.0 else scale, dtype=dtype))
        assert got["count"] == 0 and got["nonfinite"] == 6 and got["p99_9"] == 0.0

"""qsa_gather_attn_splitk_noalloc against the ordinary split-K calls (GPU).

The no-allocation entry point exists for callers that own only their inputs and outputs
and may not allocate device memory (e.g. a plugin inside a host engine that forbids
cudaMalloc while serving). It keeps the split partials in the library's static device
scratch instead of caller workspace. Its results must match the existing pair of calls
(qsa_gather_attn with num_splits > 1, then qsa_splitk_merge) within the attention tolerance,
and a second call must not see anything left over from the first -- so two different calls
run back to back on the shared scratch.

This file is named so pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

from gen import e4m3_splitk_layer, small_random
from harness import GpuPool, assert_close, bf16_dev

pytestmark = pytest.mark.gpu


def _existing(pool, wl, P):
    out, lse, _, _ = pool.attend(wl, num_splits=P)
    return out, lse


def _noalloc_via_cabi(pool, wl, P):
    """Call the new entry point through the raw C ABI (ctypes), inputs/outputs only."""
    import quantized_kv_cache_write_gb300 as q
    qd = bf16_dev(wl.q)
    idx = torch.from_numpy(np.ascontiguousarray(wl.topk, dtype=np.int32)).cuda()
    R, Hq, D = qd.shape
    out = torch.full((R, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((R, Hq), float("nan"), dtype=torch.float32, device="cuda")
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    st = q.lib.qsa_gather_attn_splitk_noalloc(
        ptr(qd), R, Hq, wl.num_kv_heads, D, pool.code, ptr(pool.k_cache), ptr(pool.v_cache),
        ptr(pool.k_scale_tok), ptr(pool.v_scale_tok), float(pool.k_scale_layer), float(pool.v_scale_layer),
        wl.num_slots, ptr(idx), wl.topk.shape[1], float(wl.softmax_scale), P, ptr(out), ptr(lse), None,
        torch.cuda.current_stream().cuda_stream)
    assert st == q.QKV_OK, q.status_str(st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


def test_noalloc_matches_existing_split_calls_twice_in_a_row():
    # call 1: calibrated E4M3, top-k 2051 in 8 splits (64 x 8 x 16 partials, ~8.4 MB)
    wl1 = e4m3_splitk_layer(0)
    pool1 = GpuPool(wl1, "e4m3")
    # call 2: int8 side, fewer rows but more splits and padding (different scratch footprint)
    wl2 = small_random(61, num_slots=20000, rows=37, topk=900, pad_frac=0.2, outlier_frac=0.01)
    pool2 = GpuPool(wl2, "int8_side")

    ref1 = _existing(pool1, wl1, 8)
    ref2 = _existing(pool2, wl2, 13)
    got1 = _noalloc_via_cabi(pool1, wl1, 8)
    got2 = _noalloc_via_cabi(pool2, wl2, 13)
    for got, ref, name in [(got1, ref1, "e4m3 P=8"), (got2, ref2, "int8 P=13")]:
        assert_close(got[0], ref[0], f"noalloc out ({name})")
        assert_close(got[1], ref[1], f"noalloc lse ({name})")
    # and once more in the first shape after the second overwrote the scratch
    again = _noalloc_via_cabi(pool1, wl1, 8)
    assert_close(again[0], ref1[0], "noalloc out (repeat)")


def test_noalloc_rejects_calls_beyond_the_scratch():
    import quantized_kv_cache_write_gb300 as q
    wl = small_random(62, num_slots=1000, rows=2, topk=10)
    pool = GpuPool(wl, "int8_side")
    rows, P, Hq = 2048, 16, 16  # 2048 x 16 x 16 x 1028 B >> 16 MiB
    assert q.noalloc_scratch_bytes(rows, P, Hq) > q.NOALLOC_SCRATCH_BYTES
    out = torch.zeros((rows, Hq, 256), dtype=torch.float32, device="cuda")
    qd = torch.zeros((rows, Hq, 256), dtype=torch.bfloat16, device="cuda")
    idx = torch.full((rows, 8), -1, dtype=torch.int32, device="cuda")
    st = q.lib.qsa_gather_attn_splitk_noalloc(
        qd.data_ptr(), rows, Hq, 1, 256, q.QKV_INT8_SIDE, pool.k_cache.data_ptr(), pool.v_cache.data_ptr(),
        pool.k_scale_tok.data_ptr(), pool.v_scale_tok.data_ptr(), 1.0, 1.0, wl.num_slots, idx.data_ptr(), 8,
        0.0625, P, out.data_ptr(), None, None, torch.cuda.current_stream().cuda_stream)
    assert st == q.QKV_ERR_ARG
    with pytest.raises(ValueError, match="static scratch"):
        q.qsa_gather_attn_splitk_noalloc(qd, q.QKV_INT8_SIDE, pool.k_cache, pool.v_cache, idx, 0.0625,
                                         num_splits=P, out=out, k_scale_tok=pool.k_scale_tok,
                                         v_scale_tok=pool.v_scale_tok)
    torch.cuda.synchronize()
    assert torch.all(out == 0)  # nothing was launched

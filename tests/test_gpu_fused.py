"""qsa_gather_attn_splitk_fused: split-K gather with the merge done by the last split CTA of
each (row, KV head), in the same launch (GPU).

"[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache" §Implementation scope (split-K workspace
and merge) and "[Perf][SM70][FP8] Hoist QSA E4M3 KV scales" §Changes (V scale once, after the
merge). The fused call runs the merge arithmetic of qsa_splitk_merge on the same partials, so
its output must equal the two-launch path bit for bit, and the oracle within the tolerance.
The arrival counters must come back zero after every call.
"""

import numpy as np
import pytest
import torch

from gen import e4m3_splitk_layer, long_context_decode, small_random
from harness import GpuPool, OraclePool, assert_close, bf16_dev

pytestmark = pytest.mark.gpu
FORMATS = ["int8_side", "int8_inline", "e4m3", "bf16"]


def _fused(gp, wl, P, counters=None, with_lse=True, dev_status=None):
    import quantized_kv_cache_write_gb300 as q
    qd = bf16_dev(wl.q)
    idx = torch.from_numpy(np.ascontiguousarray(wl.topk, dtype=np.int32)).cuda()
    R, Hq, D = qd.shape
    if counters is None:
        chunks = (Hq // wl.num_kv_heads + 15) // 16
        counters = torch.zeros((R, wl.num_kv_heads, chunks), dtype=torch.int32, device="cuda")
    out = torch.full((R, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((R, Hq), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    o_part = torch.full((R, P, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    lse_part = torch.full((R, P, Hq), float("nan"), dtype=torch.float32, device="cuda")
    q.qsa_gather_attn_splitk_fused(qd, gp.code, gp.k_cache, gp.v_cache, idx, wl.softmax_scale, num_splits=P,
                                   out=out, lse=lse, o_part=o_part, lse_part=lse_part, counters=counters,
                                   num_kv_heads=wl.num_kv_heads, num_slots=wl.num_slots,
                                   k_scale_tok=gp.k_scale_tok, v_scale_tok=gp.v_scale_tok,
                                   k_scale_layer=float(gp.k_scale_layer), v_scale_layer=float(gp.v_scale_layer),
                                   dev_status=dev_status)
    torch.cuda.synchronize()
    return (out.cpu().numpy(), lse.cpu().numpy() if with_lse else None, o_part.cpu().numpy(),
            lse_part.cpu().numpy(), counters)


def _same(a, b, what):
    assert a.shape == b.shape, what
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), f"{what}: not bit-identical"


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("P", [2, 8, 13, 64])
def test_fused_equals_two_launches_and_oracle(fmt, P):
    wl = small_random(61, num_slots=4000, rows=6, topk=515, pad_frac=0.05, outlier_frac=0.01)
    wl.topk[2] = -1  # an all-empty row: every split empty
    gp = GpuPool(wl, fmt)
    out, lse, o_part, lse_part, counters = _fused(gp, wl, P)
    ref = gp.attend(wl, num_splits=P)
    _same(out, ref[0], "out")
    _same(lse, ref[1], "lse")
    _same(o_part, ref[2], "o_part")
    _same(lse_part, ref[3], "lse_part")
    assert int(counters.abs().sum().item()) == 0
    ro, rl = OraclePool(wl, fmt).attend(wl)
    assert_close(out, ro, f"{fmt} fused out")
    assert_close(lse, rl, f"{fmt} fused lse")
    assert np.all(out[2] == 0) and np.all(lse[2] == -np.inf)


def test_counters_are_reused_across_calls_and_kv_heads():
    wl = small_random(62, num_slots=3000, rows=5, topk=300, num_q_heads=32, num_kv_heads=2, pad_frac=0.1)
    gp = GpuPool(wl, "int8_side")
    counters = torch.zeros((wl.rows, 2), dtype=torch.int32, device="cuda")
    first = _fused(gp, wl, 5, counters=counters)
    second = _fused(gp, wl, 5, counters=counters)
    _same(first[0], second[0], "out, second call")
    _same(first[1], second[1], "lse, second call")
    assert int(counters.abs().sum().item()) == 0
    ro, rl = OraclePool(wl, "int8_side").attend(wl)
    assert_close(second[0], ro, "out")
    assert_close(second[1], rl, "lse")


@pytest.mark.parametrize("hq,hkv", [(32, 1), (40, 2)])
def test_fused_with_head_chunks(hq, hkv):
    wl = small_random(64, num_slots=3000, rows=4, topk=400, num_q_heads=hq, num_kv_heads=hkv, pad_frac=0.05)
    gp = GpuPool(wl, "int8_side")
    out, lse, o_part, lse_part, counters = _fused(gp, wl, 6)
    ref = gp.attend(wl, num_splits=6)
    _same(out, ref[0], "out")
    _same(lse, ref[1], "lse")
    assert int(counters.abs().sum().item()) == 0
    ro, rl = OraclePool(wl, "int8_side").attend(wl)
    assert_close(out, ro, "out")


def test_lse_is_optional_and_single_split_runs_unsplit():
    import quantized_kv_cache_write_gb300 as q
    wl = small_random(63, num_slots=2000, rows=3, topk=100)
    gp = GpuPool(wl, "e4m3")
    out, lse, *_ = _fused(gp, wl, 4, with_lse=False)
    ro, _ = OraclePool(wl, "e4m3").attend(wl)
    assert lse is None
    assert_close(out, ro, "out without lse")
    # num_splits = 1: no workspace and no counters needed, same result as qsa_gather_attn
    qd = bf16_dev(wl.q)
    idx = torch.from_numpy(np.ascontiguousarray(wl.topk, dtype=np.int32)).cuda()
    o1 = torch.empty((3, 16, 256), dtype=torch.float32, device="cuda")
    q.qsa_gather_attn_splitk_fused(qd, gp.code, gp.k_cache, gp.v_cache, idx, wl.softmax_scale, num_splits=1,
                                   out=o1, o_part=None, lse_part=None, counters=None,
                                   k_scale_layer=float(gp.k_scale_layer), v_scale_layer=float(gp.v_scale_layer))
    torch.cuda.synchronize()
    _same(o1.cpu().numpy(), gp.attend(wl)[0], "unsplit out")


def test_e4m3_splitk_layer_fused():
    """Calibrated E4M3, top-k 2051 split 8 ways, V scale applied after the fused merge."""
    wl = e4m3_splitk_layer(0)
    gp = GpuPool(wl, "e4m3")
    out, lse, *_ , counters = _fused(gp, wl, 8)
    ref = gp.attend(wl, num_splits=8)
    _same(out, ref[0], "out")
    ro, rl = OraclePool(wl, "e4m3").attend(wl)
    assert_close(out, ro, "out")
    assert_close(lse, rl, "lse")


def test_long_context_decode_fused():
    wl = long_context_decode(3)
    gp = GpuPool(wl, "int8_side")
    out, lse, *_ = _fused(gp, wl, wl.num_splits)
    ro, rl = OraclePool(wl, "int8_side").attend(wl)
    assert_close(out, ro, "out")
    assert_close(lse, rl, "lse")


def test_suggested_split_counts():
    import quantized_kv_cache_write_gb300 as q
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # occupancy 3, 3, 3, 2 CTAs per SM (int8 side, E4M3, int8 inline, bf16), capped at 2
    for fmt, per_sm in (("int8_side", 2), ("e4m3", 2), ("int8_inline", 2), ("bf16", 2)):
        code = q.FORMATS[fmt]
        # 40 decode rows x top-k 2048: one wave of resident CTAs
        assert q.qsa_suggest_num_splits(code, 40, 16, 1, 2048) == max(1, min(16, sms * per_sm // 40))
        assert q.qsa_suggest_num_splits(code, 20, 32, 1, 2048) == max(1, min(16, sms * per_sm // 40))
        assert q.qsa_suggest_num_splits(code, 4, 16, 1, 100) == 1  # at least 128 keys per split
        assert q.qsa_suggest_num_splits(code, 100000, 16, 1, 1024) == 1  # the rows already fill the GPU

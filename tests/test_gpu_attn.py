"""GPU parity of the top-k gather decode attention and the split-K merge against the fp64
oracle, within |gpu - ref| <= 5e-5 + 1e-3 |ref| (outputs and lse).

Covers every slot-pool layout, split and unsplit launches, ragged tails, padding, empty
rows, GQA groups 8 and 16, two KV heads, and the five workload shapes of the pages
("int8 per-(token,head) KV cache for the Qwen3.8-Flash-Next QSA path" §The finding worth
upstreaming: 2048 rows x top-k 1024; "[Perf][SM70][FP8] Hoist QSA E4M3 KV scales"
§Combined SM70 validation provenance: top-k 2051 split-K; MTP decode and chunked prefill).
"""

import numpy as np
import pytest
import torch

from gen import (E4M3_SPLITK_LAYERS, chunked_prefill, e4m3_splitk_layer, long_context_decode,
                 page1_shape, small_random, tiny)
from harness import GpuPool, OraclePool, assert_close, bf16_dev
from oracle import attention as oatt

pytestmark = pytest.mark.gpu
FORMATS = ["int8_side", "int8_inline", "e4m3", "bf16"]


def _check(wl, fmt, num_splits=1, rows=None, check_parts=True):
    gp = GpuPool(wl, fmt)
    op = OraclePool(wl, fmt)
    out, lse, o_part, lse_part = gp.attend(wl, num_splits=num_splits)
    sel = slice(None) if rows is None else np.asarray(rows)
    ro, rl = op.attend(wl, rows=None if rows is None else rows)
    assert_close(out[sel], ro[sel], f"{fmt} out")
    assert_close(lse[sel], rl[sel], f"{fmt} lse")
    if num_splits > 1 and check_parts:
        po, pl = op.attend_splits(wl, num_splits, rows=None if rows is None else rows)
        assert_close(o_part[sel], po[sel], f"{fmt} o_part")
        assert_close(lse_part[sel], pl[sel], f"{fmt} lse_part")
    return out, lse


@pytest.mark.parametrize("fmt", FORMATS)
def test_tiny_config(fmt):
    _check(tiny(0), fmt)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("shape", [
    dict(topk=67, rows=9, pad_frac=0.0),          # ragged tail (67 = 64 + 3)
    dict(topk=300, rows=7, pad_frac=0.3),         # padding spread through the list
    dict(topk=1, rows=5, pad_frac=0.0),           # a single key: o = V_j
    dict(topk=2500, rows=3, pad_frac=0.1),        # several index chunks (> 1024 columns)
])
def test_ragged_and_padded(fmt, shape):
    wl = small_random(41, num_slots=6000, num_tokens=5000, outlier_frac=0.02, **shape)
    _check(wl, fmt)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("P", [2, 8, 13])
def test_split_k_partials_and_merge(fmt, P):
    wl = small_random(42, num_slots=4000, rows=6, topk=515, pad_frac=0.05, outlier_frac=0.01)
    _check(wl, fmt, num_splits=P)


@pytest.mark.parametrize("fmt", ["int8_side", "e4m3"])
def test_gqa8_and_two_kv_heads(fmt):
    _check(small_random(43, num_slots=3000, rows=5, topk=200, num_q_heads=8, num_kv_heads=1), fmt)
    _check(small_random(44, num_slots=3000, rows=5, topk=200, num_q_heads=32, num_kv_heads=2), fmt)
    _check(small_random(45, num_slots=3000, rows=4, topk=100, num_q_heads=6, num_kv_heads=2), fmt)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("hq,hkv", [(32, 1), (20, 1), (4, 1), (64, 2), (128, 1)])
def test_gqa_groups_beyond_and_below_16(fmt, hq, hkv):
    # groups above 16 run one CTA per 16 query heads (the last chunk ragged for 20)
    wl = small_random(52, num_slots=3000, rows=3, topk=150, num_q_heads=hq, num_kv_heads=hkv, pad_frac=0.1,
                      outlier_frac=0.02)
    _check(wl, fmt)
    if hq // hkv > 16:
        _check(wl, fmt, num_splits=3)


@pytest.mark.parametrize("fmt", FORMATS)
def test_outlier_heavy_seed_sweep(fmt):
    # Rows dominated by a few 16x outlier keys, the rest of the weight spread thin: the regime
    # where the small keys' p.V operands sit lowest in fp16's range. Twelve seeds, 2 - 5 %
    # outlier tokens, top-k from 64 to 1024.
    for seed in range(12):
        wl = small_random(300 + seed, num_slots=4000, rows=4, topk=64 + 80 * seed, pad_frac=0.05,
                          outlier_frac=0.02 + 0.0025 * seed)
        _check(wl, fmt)


@pytest.mark.parametrize("fmt", FORMATS)
def test_empty_rows_and_zero_topk(fmt):
    wl = small_random(46, num_slots=2000, rows=4, topk=50)
    wl.topk[1] = -1
    out, lse = _check(wl, fmt)
    assert np.all(out[1] == 0) and np.all(lse[1] == -np.inf)
    # split with empty trailing splits and an all-empty row
    _check(wl, fmt, num_splits=64)
    wl0 = small_random(47, num_slots=100, rows=3, topk=0)
    out, lse, _, _ = GpuPool(wl0, fmt).attend(wl0)
    assert np.all(out == 0) and np.all(lse == -np.inf)


def test_inline_and_side_give_bit_identical_outputs():
    wl = small_random(48, num_slots=8000, rows=8, topk=700, pad_frac=0.1, outlier_frac=0.02)
    a = GpuPool(wl, "int8_side").attend(wl)
    b = GpuPool(wl, "int8_inline").attend(wl)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_bad_indices_are_flagged_and_treated_as_padding():
    wl = small_random(49, num_slots=2000, rows=3, topk=40)
    idx = wl.topk.copy()
    idx[0, 5] = 2000
    idx[2, 0] = -9
    gp = GpuPool(wl, "int8_side")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, _, _ = gp.attend(wl, idx_dev=torch.from_numpy(idx).cuda(), dev_status=status)
    assert status.item() == 2
    clean = idx.copy()
    clean[clean >= 2000] = -1
    clean[clean < -1] = -1
    op = OraclePool(wl, "int8_side")
    ro, rl = oatt.gather_attention(wl.q, op.K, op.V, clean, wl.softmax_scale)
    assert_close(out, ro, "out")
    assert_close(lse, rl, "lse")


@pytest.mark.parametrize("fmt", FORMATS)
def test_empty_pool_gives_empty_rows_and_flags_indices(fmt):
    # the buffers hold slots, but the call says the pool is empty: every index is out of range
    import dataclasses
    wl = small_random(51, num_slots=64, rows=3, topk=40, pad_frac=0.3)
    gp = GpuPool(wl, fmt)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, _, _ = gp.attend(dataclasses.replace(wl, num_slots=0), dev_status=status)
    assert np.all(out == 0) and np.all(lse == -np.inf)
    assert status.item() == 2
    # all-padding rows with an empty pool raise nothing
    status.zero_()
    wl_pad = dataclasses.replace(wl, num_slots=0, topk=np.full_like(wl.topk, -1))
    out, lse, _, _ = gp.attend(wl_pad, dev_status=status)
    assert np.all(out == 0) and np.all(lse == -np.inf) and status.item() == 0


def test_duplicate_indices_count_twice():
    wl = small_random(50, num_slots=500, rows=2, topk=30)
    wl.topk[:, 10:20] = wl.topk[:, 0:10]
    _check(wl, "int8_side")


# ------------------------------------------------------------------ the pages' workload shapes

@pytest.fixture(scope="module")
def page1():
    return page1_shape(1, with_step=False)


@pytest.mark.parametrize("fmt", FORMATS)
def test_page1_shape_full_size_every_row(page1, fmt):
    """2048 rows x top-k 1024 over 262144 slots, launched as the benchmark launches it; every
    one of the 2048 rows (all 16 heads, all 256 dims and the lse) checked against the oracle."""
    _check(page1, fmt)


def test_e4m3_splitk_12_layers():
    """Calibrated E4M3, top-k 2051 split 8 ways (257 x 7 + 252), V scale after the merge."""
    for layer in range(E4M3_SPLITK_LAYERS):
        wl = e4m3_splitk_layer(layer)
        _check(wl, "e4m3", num_splits=8, check_parts=(layer == 0))


def test_long_context_decode_all_rows():
    wl = long_context_decode(3)
    _check(wl, "int8_side", num_splits=wl.num_splits)


def test_chunked_prefill_rows():
    """8192 causal rows launched at once; every 16th row plus the edges of the causal ramp
    (empty row 0, 1 key, the 1023 / 1024 / 1025 transition to a full top-k) checked."""
    wl = chunked_prefill(4)
    edges = np.array([0, 1, 2, 63, 64, 65, 1000, 1023, 1024, 1025, 4095, 4096, 8191])
    rows = np.union1d(np.arange(0, wl.rows, 16), edges)
    for fmt in ["int8_side", "e4m3"]:
        out, lse = _check(wl, fmt, rows=rows)
        assert np.all(out[0] == 0) and np.all(lse[0] == -np.inf)


def test_merge_kernel_against_oracle_on_random_partials():
    import quantized_kv_cache_write_gb300 as q
    rng = np.random.default_rng(51)
    R, P, Hq, D = 7, 9, 16, 256
    op = rng.standard_normal((R, P, Hq, D)).astype(np.float32)
    lp = (rng.standard_normal((R, P, Hq)) * 5).astype(np.float32)
    lp[rng.random((R, P, Hq)) < 0.2] = -np.inf
    lp[3] = -np.inf  # all-empty row
    out = torch.empty((R, Hq, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
    q.qsa_splitk_merge(torch.from_numpy(op).cuda(), torch.from_numpy(lp).cuda(), out, lse, v_scale_post=0.37)
    ro, rl = oatt.merge_splits(op.astype(np.float64), lp.astype(np.float64), v_scale_post=0.37)
    assert_close(out.cpu().numpy(), ro, "merge out", atol=1e-6, rtol=1e-5)
    assert_close(lse.cpu().numpy(), rl, "merge lse", atol=1e-6, rtol=1e-5)

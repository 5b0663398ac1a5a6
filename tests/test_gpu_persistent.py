"""The persistent grid (QSA_ENGINE_PERSISTENT): resident CTAs taking work items from a counter.

Each work item (row, KV head, 16-head chunk, split) runs the same arithmetic as its own CTA of
the default grid, so every output and partial must equal the default engine's bit for bit, and
the scheduling counter must be zero again after each launch. The mixed batches of "[Model][SM70]
[FP8] Add calibrated E4M3 QSA KV cache" (§Implementation scope: mixed catch-up/decode batches,
tails of at most 16 rows; §Targeted mixed-batch scheduler regression: 46 catch-up rows plus
three decode rows) are also checked against the fp64 oracle, |gpu - ref| <= 5e-5 + 1e-3 |ref|.
"""

import dataclasses

import numpy as np
import pytest
import torch

from gen import bulk_tail_decode, mixed_catchup_decode, small_paged, small_random
from harness import GpuPool, OraclePool, act_dev, assert_close
from oracle import attention as oatt
from oracle.paging import paged_slots

pytestmark = pytest.mark.gpu
FORMATS = ["int8_side", "int8_inline", "e4m3", "bf16"]


def _run(gp, wl, engine, P=1, fused=True, idx=None, lens=None, paged=None, sched=None, q_dev=None):
    """One qsa_gather_attn_ex call; returns out, lse, o_part, lse_part (numpy) and the status."""
    import quantized_kv_cache_write_gb300 as q
    R, Hq, D, H = wl.rows, wl.num_q_heads, wl.head_dim, wl.num_kv_heads
    out = torch.full((R, Hq, D), float("nan"), dtype=torch.float32, device="cuda") if (P == 1 or fused) else None
    lse = torch.full((R, Hq), float("nan"), dtype=torch.float32, device="cuda") if (P == 1 or fused) else None
    o_part = torch.full((R, P, Hq, D), float("nan"), dtype=torch.float32, device="cuda") if P > 1 else None
    lse_part = torch.full((R, P, Hq), float("nan"), dtype=torch.float32, device="cuda") if P > 1 else None
    counters = torch.zeros((R, H, (Hq // H + 15) // 16), dtype=torch.int32, device="cuda") if P > 1 and fused \
        else None
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = wl.topk if idx is None else idx
    kw = {}
    if paged is not None:
        table, rs, bs = paged
        kw = dict(block_table=torch.from_numpy(table).cuda(), row_seq=torch.from_numpy(rs).cuda(), block_size=bs)
    if lens is not None:
        kw["topk_len"] = torch.from_numpy(np.ascontiguousarray(lens, dtype=np.int32)).cuda()
    if engine == q.QSA_ENGINE_PERSISTENT:
        kw["sched"] = sched
    q.qsa_gather_attn_ex(act_dev(wl.q, wl.act_dtype) if q_dev is None else q_dev, gp.code, gp.k_cache, gp.v_cache,
                         torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).cuda(), wl.softmax_scale,
                         num_kv_heads=H, num_slots=wl.num_slots, k_scale_tok=gp.k_scale_tok,
                         v_scale_tok=gp.v_scale_tok, k_scale_layer=float(gp.k_scale_layer),
                         v_scale_layer=float(gp.v_scale_layer), num_splits=P, out=out, lse=lse, o_part=o_part,
                         lse_part=lse_part, counters=counters, dev_status=status, engine=engine, **kw)
    torch.cuda.synchronize()
    if counters is not None:
        assert int(counters.abs().sum().item()) == 0
    cpu = lambda t: None if t is None else t.cpu().numpy()
    return (cpu(out), cpu(lse), cpu(o_part), cpu(lse_part)), status.item()


def _same(a, b, what):
    for x, y, name in zip(a, b, ("out", "lse", "o_part", "lse_part")):
        if x is None:
            assert y is None
            continue
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32)), f"{what}: {name} differs"


def _both(gp, wl, **kw):
    import quantized_kv_cache_write_gb300 as q
    sched = torch.zeros(2, dtype=torch.int32, device="cuda")
    ref, st_ref = _run(gp, wl, q.QSA_ENGINE_DEFAULT, **kw)
    got, st = _run(gp, wl, q.QSA_ENGINE_PERSISTENT, sched=sched, **kw)
    assert st == st_ref
    assert sched.cpu().tolist() == [0, 0]  # left zero for the next launch
    again, _ = _run(gp, wl, q.QSA_ENGINE_PERSISTENT, sched=sched, **kw)
    _same(got, again, "second persistent launch")
    return ref, got


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("P,fused", [(1, False), (8, False), (8, True)])
def test_bit_identical_to_the_default_grid(fmt, P, fused):
    wl = small_random(151, num_slots=6000, rows=37, topk=700, pad_frac=0.1, outlier_frac=0.02)
    ref, got = _both(GpuPool(wl, fmt), wl, P=P, fused=fused)
    _same(ref, got, f"{fmt} P={P} fused={fused}")


@pytest.mark.parametrize("fmt", ["int8_side", "e4m3"])
def test_mixed_catchup_decode_batch(fmt):
    """46 short catch-up rows + 3 decode rows of top-k 2051, varlen, fused split-K merge."""
    wl = mixed_catchup_decode(6)
    gp = GpuPool(wl, fmt)
    ref, got = _both(gp, wl, P=8, fused=True, lens=wl.row_len)
    _same(ref, got, fmt)
    ro, rl = OraclePool(wl, fmt).attend(wl)
    assert_close(got[0], ro, f"{fmt} out")
    assert_close(got[1], rl, f"{fmt} lse")


@pytest.mark.parametrize("fmt", ["int8_side", "e4m3"])
def test_bulk_and_tail_batch(fmt):
    """48 full rows + a 13-row tail of mixed lengths, varlen, fused split-K merge."""
    wl = bulk_tail_decode(7)
    gp = GpuPool(wl, fmt)
    garbage = wl.topk.copy()
    rng = np.random.default_rng(9)
    for r in range(wl.rows):  # entries past a row's length are never read
        garbage[r, wl.row_len[r]:] = rng.integers(10 ** 6, 10 ** 9, wl.topk.shape[1] - wl.row_len[r])
    ref, got = _both(gp, wl, P=8, fused=True, lens=wl.row_len, idx=garbage)
    _same(ref, got, fmt)
    rows = list(range(0, 48, 7)) + list(range(48, 61))
    ro, rl = OraclePool(wl, fmt).attend(wl, rows=rows)
    assert_close(got[0][rows], ro[rows], f"{fmt} out")
    assert_close(got[1][rows], rl[rows], f"{fmt} lse")


@pytest.mark.parametrize("fmt", ["int8_side", "e4m3", "bf16"])
def test_paged_gqa32_and_head_dim_128(fmt):
    wl = small_paged(152, num_seqs=4, max_blocks=8, block_size=16, rows=6, topk=90, unallocated_frac=0.0)
    slots, _, _ = paged_slots(wl.block_table, wl.row_seq, wl.topk_pos, wl.block_size, wl.num_slots)
    wls = dataclasses.replace(wl, topk=slots.astype(np.int32))
    gp = GpuPool(wls, fmt)
    ref, got = _both(gp, wl, P=4, fused=True, idx=wl.topk_pos, paged=(wl.block_table, wl.row_seq, wl.block_size))
    _same(ref, got, f"{fmt} paged")
    for kw in (dict(num_q_heads=32), dict(num_q_heads=64, num_kv_heads=2), dict(head_dim=128)):
        wl = small_random(153, num_slots=3000, rows=5, topk=400, pad_frac=0.05, **kw)
        gp = GpuPool(wl, fmt)
        ref, got = _both(gp, wl, P=3, fused=True)
        _same(ref, got, f"{fmt} {kw}")


@pytest.mark.parametrize("fmt", ["int8_side", "e4m3", "f16"])
def test_fp16_query(fmt):
    wl = small_random(154, num_slots=3000, rows=9, topk=300, pad_frac=0.05, act_dtype="f16")
    gp = GpuPool(wl, fmt)
    ref, got = _both(gp, wl, P=2, fused=True)
    _same(ref, got, fmt)


def test_more_items_than_resident_ctas_and_bad_indices():
    """2048 rows x 4 splits (8192 items, several per resident CTA) with flagged entries."""
    wl = small_random(155, num_slots=20000, rows=2048, topk=96, pad_frac=0.05)
    idx = wl.topk.copy()
    idx[5, 3] = 20000
    idx[2047, 0] = -7
    gp = GpuPool(wl, "int8_side")
    ref, got = _both(gp, wl, P=4, fused=True, idx=idx)
    _same(ref, got, "many items")
    clean = np.where((idx >= 20000) | (idx < -1), -1, idx)
    op = OraclePool(wl, "int8_side")
    rows = [0, 5, 1000, 2047]
    ro, rl = oatt.gather_attention(wl.q, op.K, op.V, clean, wl.softmax_scale, rows=rows)
    assert_close(got[0][rows], ro[rows], "out")
    assert_close(got[1][rows], rl[rows], "lse")

"""The tensor-memory engine of the int8 side gather (QSA_ENGINE_TCGEN05) against the fp64 oracle.

Same operation, same tolerance as the default engine: |gpu - ref| <= 5e-5 + 1e-3 |ref| on the
outputs and the lse ("int8 per-(token,head) KV cache for the Qwen3.8-Flash-Next QSA path"
§The finding worth upstreaming). Covers ragged tails, padding, empty rows, GQA 4 / 5 / 16 with
one and two KV heads, split-K partials, rows of different lengths, flagged indices and the
2048-row x top-k 1024 shape of that page, every row.
"""

import numpy as np
import pytest
import torch

from gen import page1_shape, small_random, tiny
from harness import GpuPool, OraclePool, act_dev, assert_close
from oracle import attention as oatt

pytestmark = pytest.mark.gpu


def _attend(gp, wl, idx=None, lens=None, P=1, status=None):
    import quantized_kv_cache_write_gb300 as q
    R, Hq, D = wl.rows, wl.num_q_heads, wl.head_dim
    idx_d = torch.from_numpy(np.ascontiguousarray(wl.topk if idx is None else idx, dtype=np.int32)).cuda()
    len_d = None if lens is None else torch.from_numpy(np.ascontiguousarray(lens, dtype=np.int32)).cuda()
    out = torch.full((R, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((R, Hq), float("nan"), dtype=torch.float32, device="cuda")
    kw = dict(num_kv_heads=wl.num_kv_heads, num_slots=wl.num_slots, k_scale_tok=gp.k_scale_tok,
              v_scale_tok=gp.v_scale_tok, dev_status=status, topk_len=len_d, engine=q.QSA_ENGINE_TCGEN05)
    if P == 1:
        q.qsa_gather_attn_ex(act_dev(wl.q), q.QKV_INT8_SIDE, gp.k_cache, gp.v_cache, idx_d, wl.softmax_scale,
                             out=out, lse=lse, **kw)
        torch.cuda.synchronize()
        return out.cpu().numpy(), lse.cpu().numpy(), None, None
    o_part = torch.full((R, P, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    lse_part = torch.full((R, P, Hq), float("nan"), dtype=torch.float32, device="cuda")
    q.qsa_gather_attn_ex(act_dev(wl.q), q.QKV_INT8_SIDE, gp.k_cache, gp.v_cache, idx_d, wl.softmax_scale,
                         num_splits=P, o_part=o_part, lse_part=lse_part, **kw)
    q.qsa_splitk_merge(o_part, lse_part, out, lse)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy(), o_part.cpu().numpy(), lse_part.cpu().numpy()


def _check(wl, P=1):
    gp, op = GpuPool(wl, "int8_side"), OraclePool(wl, "int8_side")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, o_part, lse_part = _attend(gp, wl, P=P, status=status)
    assert status.item() == 0
    ro, rl = op.attend(wl)
    assert_close(out, ro, "out")
    assert_close(lse, rl, "lse")
    if P > 1:
        po, pl = op.attend_splits(wl, P)
        assert_close(o_part, po, "o_part")
        assert_close(lse_part, pl, "lse_part")
    return out, lse


def test_tiny():
    _check(tiny(0))


@pytest.mark.parametrize("kw", [dict(topk=67, rows=9), dict(topk=300, rows=7, pad_frac=0.3),
                                dict(topk=1, rows=5), dict(topk=2500, rows=3, pad_frac=0.1)])
def test_ragged_and_padded(kw):
    _check(small_random(41, num_slots=6000, num_tokens=5000, outlier_frac=0.02, **kw))


@pytest.mark.parametrize("hq,hkv", [(8, 2), (5, 1), (16, 1), (32, 2)])
def test_gqa_groups_up_to_16(hq, hkv):
    _check(small_random(43, num_slots=3000, rows=5, topk=400, num_q_heads=hq, num_kv_heads=hkv,
                        outlier_frac=0.02))


@pytest.mark.parametrize("P", [2, 8, 13])
def test_split_k_partials(P):
    _check(small_random(42, num_slots=4000, rows=6, topk=515, pad_frac=0.05, outlier_frac=0.01), P=P)


def test_outlier_seed_sweep():
    for seed in range(6):
        _check(small_random(100 + seed, num_slots=4096, rows=16, topk=1024, outlier_frac=0.05,
                            outlier_factor=20.0))


def test_empty_rows_zero_tokens_and_rows_of_different_lengths():
    wl = small_random(46, num_slots=500, rows=4, topk=40)
    wl.topk[1] = -1
    out, lse = _check(wl)
    assert np.all(out[1] == 0) and np.all(lse[1] == -np.inf)
    _check(small_random(45, num_slots=3000, rows=5, topk=400, zero_tokens=50))
    wl = small_random(131, num_slots=4000, rows=9, topk=600, pad_frac=0.05, outlier_frac=0.01)
    rng = np.random.default_rng(7)
    lens = rng.integers(0, 601, wl.rows)
    lens[0], lens[1], lens[2] = 0, 600, 1
    idx, garbage = wl.topk.copy(), wl.topk.copy()
    for r in range(wl.rows):
        garbage[r, lens[r]:] = rng.integers(10 ** 6, 10 ** 9, wl.topk.shape[1] - lens[r])  # never read
        idx[r, lens[r]:] = -1
    gp, op = GpuPool(wl, "int8_side"), OraclePool(wl, "int8_side")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for P in (1, 4):
        out, lse, _, _ = _attend(gp, wl, idx=garbage, lens=lens, P=P, status=status)
        ro, rl = oatt.gather_attention(wl.q, op.K, op.V, idx, wl.softmax_scale)
        assert_close(out, ro, f"varlen out P={P}")
        assert_close(lse, rl, f"varlen lse P={P}")
    assert status.item() == 0


def test_bad_indices_are_flagged_and_treated_as_padding():
    wl = small_random(49, num_slots=2000, rows=3, topk=40)
    idx = wl.topk.copy()
    idx[0, 5] = 2000
    idx[2, 0] = -9
    gp = GpuPool(wl, "int8_side")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, _, _ = _attend(gp, wl, idx=idx, status=status)
    assert status.item() == 2
    clean = np.where((idx >= 2000) | (idx < -1), -1, idx)
    op = OraclePool(wl, "int8_side")
    ro, rl = oatt.gather_attention(wl.q, op.K, op.V, clean, wl.softmax_scale)
    assert_close(out, ro, "out")
    assert_close(lse, rl, "lse")


def test_page1_shape_full_size_every_row():
    """2048 rows x top-k 1024 over 262144 slots, every row against the oracle."""
    _check(page1_shape(1, with_step=False))

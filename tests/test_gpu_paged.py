"""qsa_gather_attn_paged against the oracle (GPU).

The paged kernel maps each row's logical positions to slots through the block table itself.
The oracle translates them separately (oracle/paging.py), then attends over the slot ids.
Where both kernels see the same slots, the paged result must also equal qsa_gather_attn's
bit for bit: the translation is the only difference.
"""

import dataclasses

import numpy as np
import pytest
import torch

from gen import long_context_decode, small_paged
from harness import GpuPool, OraclePool, assert_close, bf16_dev
from oracle.paging import paged_slots

pytestmark = pytest.mark.gpu
FORMATS = ["int8_side", "int8_inline", "e4m3", "bf16"]


def _attend_paged(gp, wl, num_splits=1, row_seq=None, dev_status=None):
    import quantized_kv_cache_write_gb300 as q
    qd = bf16_dev(wl.q)
    R, Hq, D = qd.shape
    table = torch.from_numpy(np.ascontiguousarray(wl.block_table, dtype=np.int32)).cuda()
    rs = torch.from_numpy(np.ascontiguousarray(wl.row_seq if row_seq is None else row_seq, dtype=np.int32)).cuda()
    pos = torch.from_numpy(np.ascontiguousarray(wl.topk_pos, dtype=np.int32)).cuda()
    kw = dict(num_kv_heads=wl.num_kv_heads, num_slots=wl.num_slots, k_scale_tok=gp.k_scale_tok,
              v_scale_tok=gp.v_scale_tok, k_scale_layer=float(gp.k_scale_layer),
              v_scale_layer=float(gp.v_scale_layer), dev_status=dev_status)
    out = torch.full((R, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((R, Hq), float("nan"), dtype=torch.float32, device="cuda")
    if num_splits == 1:
        q.qsa_gather_attn_paged(qd, gp.code, gp.k_cache, gp.v_cache, table, rs, pos, wl.block_size,
                                wl.softmax_scale, out=out, lse=lse, **kw)
    else:
        P = num_splits
        o_part = torch.full((R, P, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        lse_part = torch.full((R, P, Hq), float("nan"), dtype=torch.float32, device="cuda")
        q.qsa_gather_attn_paged(qd, gp.code, gp.k_cache, gp.v_cache, table, rs, pos, wl.block_size,
                                wl.softmax_scale, num_splits=P, o_part=o_part, lse_part=lse_part, **kw)
        q.qsa_splitk_merge(o_part, lse_part, out, lse,
                           v_scale_post=float(gp.v_scale_layer) if gp.fmt == "e4m3" else 1.0)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


def _with_slots(wl, row_seq=None):
    slots, bad, bad_row = paged_slots(wl.block_table, wl.row_seq if row_seq is None else row_seq,
                                      wl.topk_pos, wl.block_size, wl.num_slots)
    return dataclasses.replace(wl, topk=slots.astype(np.int32)), bad, bad_row


@pytest.mark.parametrize("fmt", FORMATS)
def test_small_paged_pool_matches_oracle_and_flags_unallocated_blocks(fmt):
    wl = small_paged(71)
    gp = GpuPool(wl, fmt)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = _attend_paged(gp, wl, dev_status=status)
    wls, bad, _ = _with_slots(wl)
    assert bad.any(), "the fixture must exercise unallocated blocks"
    assert status.item() == 2
    ro, rl = OraclePool(wl, fmt).attend(wls)
    assert_close(out, ro, f"{fmt} out")
    assert_close(lse, rl, f"{fmt} lse")
    # same slots through the slot-id entry point: identical bits
    o2, l2, _, _ = gp.attend(wls)
    assert np.array_equal(out, o2) and np.array_equal(lse, l2)


@pytest.mark.parametrize("block_size", [12, 1, 64])
def test_block_sizes_that_are_not_sixteen(block_size):
    wl = small_paged(72, block_size=block_size, max_blocks=max(2, 96 // block_size), topk=48)
    gp = GpuPool(wl, "int8_side")
    out, lse = _attend_paged(gp, wl, num_splits=3)
    wls, _, _ = _with_slots(wl)
    ro, rl = OraclePool(wl, "int8_side").attend(wls)
    assert_close(out, ro, f"block {block_size} out")
    assert_close(lse, rl, f"block {block_size} lse")


def test_bad_positions_and_sequences_are_flagged_and_read_as_padding():
    wl = small_paged(73, unallocated_frac=0.0, pad_frac=0.0)
    pos = wl.topk_pos.copy()
    pos[0, 3] = -7                                  # below -1
    pos[1, 0] = wl.block_table.shape[1] * wl.block_size  # past the sequence's blocks
    row_seq = wl.row_seq.copy()
    row_seq[2] = 99                                 # no such sequence: the row is empty
    wl = dataclasses.replace(wl, topk_pos=pos)
    gp = GpuPool(wl, "int8_side")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = _attend_paged(gp, wl, row_seq=row_seq, dev_status=status)
    assert status.item() == 2
    wls, bad, bad_row = _with_slots(wl, row_seq)
    assert bad[0, 3] and bad[1, 0] and bad_row[2]
    assert np.all(out[2] == 0) and np.all(lse[2] == -np.inf)
    ro, rl = OraclePool(wl, "int8_side").attend(wls)
    assert_close(out, ro, "out")
    assert_close(lse, rl, "lse")


def test_long_context_decode_paged_equals_slot_ids():
    """8 sequences x 131072 tokens in blocks of 16 (random block permutation), 5 rows each,
    top-k 2048 split 16 ways: the paged kernel reproduces the slot-id kernel bit for bit, and
    the oracle's translation reproduces the generator's slot ids."""
    wl = long_context_decode(3)
    slots, bad, bad_row = paged_slots(wl.block_table, wl.row_seq, wl.topk_pos, wl.block_size, wl.num_slots)
    assert not bad.any() and not bad_row.any() and np.array_equal(slots, wl.topk.astype(np.int64))
    gp = GpuPool(wl, "int8_side")
    out, lse = _attend_paged(gp, wl, num_splits=wl.num_splits)
    o2, l2, _, _ = gp.attend(wl, num_splits=wl.num_splits)
    assert np.array_equal(out, o2) and np.array_equal(lse, l2)

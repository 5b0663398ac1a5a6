"""qsa_gather_attn_ex: the gather's options combined in one call (GPU).

Paged pools, per-row lengths, the fused split-K merge and an fp16 query, together. Each
combination must match the fp64 oracle on the translated, truncated rows within
|gpu - ref| <= 5e-5 + 1e-3 |ref|, and the plain descriptor call must equal qsa_gather_attn bit
for bit. ("[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache" §Implementation scope: paged
storage, split-K, mixed batches; §Purpose: FP16 activations.)
"""

import dataclasses

import numpy as np
import pytest
import torch

from gen import small_paged, small_random
from harness import GpuPool, OraclePool, act_dev, assert_close
from oracle import attention as oatt
from oracle.paging import paged_slots

pytestmark = pytest.mark.gpu


def _buffers(R, Hq, D, P, H=1):
    out = torch.full((R, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((R, Hq), float("nan"), dtype=torch.float32, device="cuda")
    o_part = torch.empty((R, P, Hq, D), dtype=torch.float32, device="cuda") if P > 1 else None
    lse_part = torch.empty((R, P, Hq), dtype=torch.float32, device="cuda") if P > 1 else None
    counters = torch.zeros((R, H, (Hq // H + 15) // 16), dtype=torch.int32, device="cuda") if P > 1 else None
    return out, lse, o_part, lse_part, counters


@pytest.mark.parametrize("fmt", ["int8_side", "e4m3", "bf16"])
def test_paged_varlen_fused(fmt):
    import quantized_kv_cache_write_gb300 as q
    wl = small_paged(141, num_seqs=4, max_blocks=8, block_size=16, rows=6, topk=90, unallocated_frac=0.0)
    slots, bad, bad_row = paged_slots(wl.block_table, wl.row_seq, wl.topk_pos, wl.block_size, wl.num_slots)
    rng = np.random.default_rng(3)
    lens = rng.integers(0, 91, wl.rows).astype(np.int32)
    lens[0] = 90
    slots = slots.copy()
    pos = wl.topk_pos.copy()
    for r in range(wl.rows):
        slots[r, lens[r]:] = -1
        pos[r, lens[r]:] = rng.integers(10 ** 6, 10 ** 8, 90 - lens[r])  # never read
    wls = dataclasses.replace(wl, topk=slots.astype(np.int32))
    gp = GpuPool(wls, fmt)
    R, Hq, D, P = wl.rows, wl.num_q_heads, wl.head_dim, 4
    out, lse, o_part, lse_part, counters = _buffers(R, Hq, D, P)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q.qsa_gather_attn_ex(act_dev(wl.q), gp.code, gp.k_cache, gp.v_cache, torch.from_numpy(pos).cuda(),
                         wl.softmax_scale, k_scale_tok=gp.k_scale_tok, v_scale_tok=gp.v_scale_tok,
                         k_scale_layer=float(gp.k_scale_layer), v_scale_layer=float(gp.v_scale_layer),
                         num_splits=P, out=out, lse=lse, o_part=o_part, lse_part=lse_part, counters=counters,
                         topk_len=torch.from_numpy(lens).cuda(), block_table=torch.from_numpy(wl.block_table).cuda(),
                         row_seq=torch.from_numpy(wl.row_seq).cuda(), block_size=wl.block_size, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0 and int(counters.abs().sum().item()) == 0
    ro, rl = OraclePool(wls, fmt).attend(wls)
    assert_close(out.cpu().numpy(), ro, f"{fmt} out")
    assert_close(lse.cpu().numpy(), rl, f"{fmt} lse")


@pytest.mark.parametrize("fmt", ["int8_side", "e4m3", "f16"])
def test_fp16_query_varlen_fused_gqa32(fmt):
    import quantized_kv_cache_write_gb300 as q
    wl = small_random(142, num_slots=3000, rows=5, topk=400, num_q_heads=32, pad_frac=0.05, outlier_frac=0.01,
                      act_dtype="f16")
    lens = np.array([400, 0, 17, 399, 250], dtype=np.int32)
    idx = wl.topk.copy()
    for r in range(wl.rows):
        idx[r, lens[r]:] = -1
    gp = GpuPool(wl, fmt)
    R, Hq, D, P = wl.rows, wl.num_q_heads, wl.head_dim, 3
    out, lse, o_part, lse_part, counters = _buffers(R, Hq, D, P)
    q.qsa_gather_attn_ex(act_dev(wl.q, "f16"), gp.code, gp.k_cache, gp.v_cache, torch.from_numpy(wl.topk).cuda(),
                         wl.softmax_scale, k_scale_tok=gp.k_scale_tok, v_scale_tok=gp.v_scale_tok,
                         k_scale_layer=float(gp.k_scale_layer), v_scale_layer=float(gp.v_scale_layer),
                         num_splits=P, out=out, lse=lse, o_part=o_part, lse_part=lse_part, counters=counters,
                         topk_len=torch.from_numpy(lens).cuda())
    torch.cuda.synchronize()
    op = OraclePool(wl, fmt)
    ro, rl = oatt.gather_attention(wl.q, op.K, op.V, idx, wl.softmax_scale, q_dtype="f16")
    assert_close(out.cpu().numpy(), ro, f"{fmt} out")
    assert_close(lse.cpu().numpy(), rl, f"{fmt} lse")
    assert np.all(out.cpu().numpy()[1] == 0)


def test_plain_descriptor_equals_qsa_gather_attn():
    import quantized_kv_cache_write_gb300 as q
    wl = small_random(143, num_slots=3000, rows=4, topk=300, pad_frac=0.1)
    gp = GpuPool(wl, "int8_side")
    out, lse, *_ = _buffers(wl.rows, 16, 256, 1)
    q.qsa_gather_attn_ex(act_dev(wl.q), gp.code, gp.k_cache, gp.v_cache, torch.from_numpy(wl.topk).cuda(),
                         wl.softmax_scale, k_scale_tok=gp.k_scale_tok, v_scale_tok=gp.v_scale_tok, out=out, lse=lse)
    torch.cuda.synchronize()
    ref = gp.attend(wl)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref[0].view(np.uint32))
    assert np.array_equal(lse.cpu().numpy().view(np.uint32), ref[1].view(np.uint32))

"""A pool sharded by slot range, emulated on one GPU.

Rows are independent, so the data-parallel path shards rows with no exchange. A pool too large
for one GPU would instead be split by slot range: each rank attends its row's entries that
fall in its own slots, and one exchange of the (o, lse) partials feeds the same log-sum-exp
merge the split-K path uses ("[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache"
§Implementation scope: split-K workspace and merge). The ranks are emulated here as separate
launches on one GPU -- none waits for another -- and their partials are stacked and merged
with qsa_splitk_merge. The result must equal the oracle's unsharded attention.
"""

import numpy as np
import pytest
import torch

from gen import small_random
from harness import GpuPool, OraclePool, act_dev, assert_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt", ["int8_side", "e4m3"])
@pytest.mark.parametrize("world", [2, 3])
def test_slot_range_shards_merge_to_the_unsharded_result(fmt, world):
    import quantized_kv_cache_write_gb300 as q
    wl = small_random(151, num_slots=6000, rows=6, topk=700, pad_frac=0.05, outlier_frac=0.01)
    gp = GpuPool(wl, fmt)
    R, Hq, D, S = wl.rows, wl.num_q_heads, wl.head_dim, wl.num_slots
    o_part = torch.empty((R, world, Hq, D), dtype=torch.float32, device="cuda")
    lse_part = torch.empty((R, world, Hq), dtype=torch.float32, device="cuda")
    bounds = np.linspace(0, S, world + 1).astype(int)
    for rank in range(world):
        lo, hi = bounds[rank], bounds[rank + 1]
        mine = np.where((wl.topk >= lo) & (wl.topk < hi), wl.topk, -1).astype(np.int32)  # this rank's view
        out = torch.empty((R, Hq, D), dtype=torch.float32, device="cuda")
        lse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
        q.qsa_gather_attn(act_dev(wl.q), gp.code, gp.k_cache, gp.v_cache, torch.from_numpy(mine).cuda(),
                          wl.softmax_scale, k_scale_tok=gp.k_scale_tok, v_scale_tok=gp.v_scale_tok,
                          k_scale_layer=float(gp.k_scale_layer), v_scale_layer=float(gp.v_scale_layer),
                          out=out, lse=lse)
        o_part[:, rank] = out  # the exchange: each rank's normalised partial and its lse
        lse_part[:, rank] = lse
    merged = torch.empty((R, Hq, D), dtype=torch.float32, device="cuda")
    mlse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
    q.qsa_splitk_merge(o_part, lse_part, merged, mlse)  # V scales are already inside the partials
    torch.cuda.synchronize()
    ro, rl = OraclePool(wl, fmt).attend(wl)
    assert_close(merged.cpu().numpy(), ro, f"{fmt} sharded out")
    assert_close(mlse.cpu().numpy(), rl, f"{fmt} sharded lse")


@pytest.mark.parametrize("fmt", ["int8_side", "int8_inline", "e4m3", "bf16"])
@pytest.mark.parametrize("world", [2, 3])
def test_shard_pools_hold_only_their_slot_range(fmt, world):
    """Each rank holds only its own slots, written at local ids; the gather takes the global ids
    (slot_lo / shard mode), skips other ranks' entries unflagged, and the merged partials equal
    the unsharded oracle -- and, bit for bit, the masked launches on the whole pool above."""
    import dataclasses
    import quantized_kv_cache_write_gb300 as q
    wl = small_random(161, num_slots=6000, rows=6, topk=700, pad_frac=0.05, outlier_frac=0.01)
    full = GpuPool(wl, fmt)
    R, Hq, D, S = wl.rows, wl.num_q_heads, wl.head_dim, wl.num_slots
    o_part = torch.empty((R, world, Hq, D), dtype=torch.float32, device="cuda")
    lse_part = torch.empty((R, world, Hq), dtype=torch.float32, device="cuda")
    bounds = np.linspace(0, S, world + 1).astype(int)
    idx = torch.from_numpy(np.ascontiguousarray(wl.topk, dtype=np.int32)).cuda()
    for rank in range(world):
        lo, hi = int(bounds[rank]), int(bounds[rank + 1])
        sm = wl.slot_mapping
        local = dataclasses.replace(wl, num_slots=hi - lo, slot_mapping=np.where((sm >= lo) & (sm < hi), sm - lo, -1))
        gp = GpuPool(local, fmt)
        if fmt == "e4m3":  # one calibrated scale per layer, whatever the shard
            assert (gp.k_scale_layer, gp.v_scale_layer) == (full.k_scale_layer, full.v_scale_layer)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.empty((R, Hq, D), dtype=torch.float32, device="cuda")
        lse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
        q.qsa_gather_attn_ex(act_dev(wl.q), gp.code, gp.k_cache, gp.v_cache, idx, wl.softmax_scale,
                             num_slots=hi - lo, k_scale_tok=gp.k_scale_tok, v_scale_tok=gp.v_scale_tok,
                             k_scale_layer=float(gp.k_scale_layer), v_scale_layer=float(gp.v_scale_layer),
                             out=out, lse=lse, dev_status=status, slot_lo=lo)
        # the same partial from a masked launch on the whole pool
        mine = np.where((wl.topk >= lo) & (wl.topk < hi), wl.topk, -1).astype(np.int32)
        ref_o = torch.empty_like(out)
        ref_l = torch.empty_like(lse)
        q.qsa_gather_attn(act_dev(wl.q), full.code, full.k_cache, full.v_cache, torch.from_numpy(mine).cuda(),
                          wl.softmax_scale, k_scale_tok=full.k_scale_tok, v_scale_tok=full.v_scale_tok,
                          k_scale_layer=float(full.k_scale_layer), v_scale_layer=float(full.v_scale_layer),
                          out=ref_o, lse=ref_l)
        torch.cuda.synchronize()
        assert status.item() == 0  # other ranks' entries are not errors
        assert torch.equal(out.view(torch.int32), ref_o.view(torch.int32))
        assert torch.equal(lse.view(torch.int32), ref_l.view(torch.int32))
        o_part[:, rank] = out
        lse_part[:, rank] = lse
    merged = torch.empty((R, Hq, D), dtype=torch.float32, device="cuda")
    mlse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
    q.qsa_splitk_merge(o_part, lse_part, merged, mlse)
    torch.cuda.synchronize()
    ro, rl = OraclePool(wl, fmt).attend(wl)
    assert_close(merged.cpu().numpy(), ro, f"{fmt} shard-mode out")
    assert_close(mlse.cpu().numpy(), rl, f"{fmt} shard-mode lse")

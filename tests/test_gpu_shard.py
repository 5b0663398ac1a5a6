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

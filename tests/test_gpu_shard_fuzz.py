"""Seeded random slot-range shards against the fp64 oracle (GPU).

Each case draws a pool layout, head dim, GQA group, KV-head count, rows, top-k width, per-row
lengths (or none), a shard count (2 or 3), and per shard a split count with the fused or the
separate merge. The pool's global slots are cut into contiguous ranges; each shard holds its
range at local ids (written by the library from the same tokens, so an E4M3 shard calibrates
the same per-layer scales) and gathers the rows' global entries in shard mode, skipping other
shards' entries. qsa_splitk_merge over the shards' (output, lse) partials must give the oracle's
attention over the whole pool, within |gpu - ref| <= 5e-5 + 1e-3 |ref|, with nothing flagged.
("[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache" §Implementation scope: split-K
partials and their merge.)
"""

import dataclasses

import numpy as np
import pytest
import torch

from gen import small_random
from harness import GpuPool, OraclePool, act_dev, assert_close

pytestmark = pytest.mark.gpu


def _draw(seed):
    rng = np.random.default_rng([9431, seed])
    return dict(fmt=str(rng.choice(["int8_side", "int8_inline", "e4m3", "bf16"])), hd=int(rng.choice([128, 256])),
                hkv=int(rng.choice([1, 1, 2])), g=int(rng.choice([1, 8, 16, 16, 20])), rows=int(rng.integers(1, 10)),
                topk=int(rng.choice([1, 17, 100, 700])), varlen=bool(rng.integers(2)),
                shards=int(rng.choice([2, 3])), P=[int(p) for p in rng.choice([1, 1, 2, 4], size=3)],
                fused=[bool(f) for f in rng.integers(0, 2, size=3)], seed=int(rng.integers(1 << 30)))


@pytest.mark.parametrize("case", range(24))
def test_random_shards_merge_to_the_whole_pool(case):
    import quantized_kv_cache_write_gb300 as q
    c = _draw(case)
    wl = small_random(c["seed"], num_slots=3000, rows=c["rows"], topk=c["topk"], num_q_heads=c["g"] * c["hkv"],
                      num_kv_heads=c["hkv"], pad_frac=0.05, outlier_frac=0.02, head_dim=c["hd"])
    R, Hq, D, S = wl.rows, wl.num_q_heads, wl.head_dim, wl.num_slots
    lens = np.random.default_rng(c["seed"]).integers(0, c["topk"] + 1, R).astype(np.int32) if c["varlen"] else None
    ref_idx = wl.topk.copy()
    if lens is not None:
        for r in range(R):
            ref_idx[r, lens[r]:] = -1
    idx = torch.from_numpy(np.ascontiguousarray(wl.topk, dtype=np.int32)).cuda()
    qd = act_dev(wl.q)
    bounds = np.linspace(0, S, c["shards"] + 1).astype(np.int64)
    o_sh = torch.empty((R, c["shards"], Hq, D), dtype=torch.float32, device="cuda")
    l_sh = torch.empty((R, c["shards"], Hq), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for s in range(c["shards"]):
        lo, hi = int(bounds[s]), int(bounds[s + 1])
        sm = wl.slot_mapping
        local = dataclasses.replace(wl, num_slots=hi - lo, slot_mapping=np.where((sm >= lo) & (sm < hi), sm - lo, -1))
        gp = GpuPool(local, c["fmt"])
        P, fused = c["P"][s], c["fused"][s]
        out = torch.empty((R, Hq, D), dtype=torch.float32, device="cuda")
        lse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
        kw = dict(num_kv_heads=c["hkv"], num_slots=hi - lo, k_scale_tok=gp.k_scale_tok, v_scale_tok=gp.v_scale_tok,
                  k_scale_layer=float(gp.k_scale_layer), v_scale_layer=float(gp.v_scale_layer), dev_status=status,
                  topk_len=None if lens is None else torch.from_numpy(lens).cuda(), slot_lo=lo)
        if P == 1:
            q.qsa_gather_attn_ex(qd, gp.code, gp.k_cache, gp.v_cache, idx, wl.softmax_scale, out=out, lse=lse, **kw)
        else:
            o_part = torch.empty((R, P, Hq, D), dtype=torch.float32, device="cuda")
            lse_part = torch.empty((R, P, Hq), dtype=torch.float32, device="cuda")
            if fused:
                counters = torch.zeros((R, c["hkv"], (c["g"] + 15) // 16), dtype=torch.int32, device="cuda")
                q.qsa_gather_attn_ex(qd, gp.code, gp.k_cache, gp.v_cache, idx, wl.softmax_scale, num_splits=P,
                                     out=out, lse=lse, o_part=o_part, lse_part=lse_part, counters=counters, **kw)
            else:
                q.qsa_gather_attn_ex(qd, gp.code, gp.k_cache, gp.v_cache, idx, wl.softmax_scale, num_splits=P,
                                     o_part=o_part, lse_part=lse_part, **kw)
                q.qsa_splitk_merge(o_part, lse_part, out, lse,
                                   v_scale_post=float(gp.v_scale_layer) if c["fmt"] == "e4m3" else 1.0)
        o_sh[:, s] = out
        l_sh[:, s] = lse
    merged = torch.empty((R, Hq, D), dtype=torch.float32, device="cuda")
    mlse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
    q.qsa_splitk_merge(o_sh, l_sh, merged, mlse)  # each shard's output already carries the V scale
    torch.cuda.synchronize()
    assert status.item() == 0, c
    wlr = dataclasses.replace(wl, topk=ref_idx)
    ro, rl = OraclePool(wlr, c["fmt"]).attend(wlr)
    assert_close(merged.cpu().numpy(), ro, f"out {c}")
    assert_close(mlse.cpu().numpy(), rl, f"lse {c}")

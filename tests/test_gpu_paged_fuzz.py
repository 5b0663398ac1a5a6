"""Seeded random paged gathers against the fp64 oracle (GPU).

Each case draws a pool layout, head dim, GQA group, KV-head count, block size, sequence count
and blocks per sequence (some table entries unallocated), rows with padding and (or not)
per-row lengths, a split count with the fused or the separate merge, and the default or the
persistent engine. The kernel maps each row's positions through the block table itself; the
oracle translates them separately (oracle/paging.py) and attends over the slot ids. Every
output and lse element within |gpu - ref| <= 5e-5 + 1e-3 |ref|, and the status word flags
exactly the cases with a position in an unallocated block inside a row's length. The draws are
seeded, so a failure names a reproducible configuration.
("[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache" §Implementation scope: the paged
("page4") KV layout the decode kernels read.)
"""

import dataclasses

import numpy as np
import pytest
import torch

from gen import small_paged
from harness import GpuPool, OraclePool, act_dev, assert_close
from oracle.paging import paged_slots

pytestmark = pytest.mark.gpu


def _draw(seed):
    rng = np.random.default_rng([5150, seed])
    fmt = str(rng.choice(["int8_side", "int8_inline", "e4m3", "bf16"]))
    bs = int(rng.choice([1, 12, 16, 16, 64]))
    max_blocks = max(1, int(rng.integers(64, 1600)) // bs)
    P = int(rng.choice([1, 1, 2, 5]))
    return dict(fmt=fmt, hd=int(rng.choice([128, 256])), hkv=int(rng.choice([1, 1, 2])),
                g=int(rng.choice([1, 8, 16, 16, 20, 32])), bs=bs, seqs=int(rng.integers(1, 5)),
                max_blocks=max_blocks, rows=int(rng.integers(1, 13)),
                topk=int(min(rng.choice([1, 17, 100, 700]), max_blocks * bs)),
                pad=float(rng.choice([0.0, 0.1])), unalloc=float(rng.choice([0.0, 0.0, 0.1])), P=P,
                fused=bool(rng.integers(2)) and P > 1, varlen=bool(rng.integers(2)),
                persistent=bool(rng.integers(3) == 0), seed=int(rng.integers(1 << 30)))


@pytest.mark.parametrize("case", range(40))
def test_random_paged_configuration(case):
    import quantized_kv_cache_write_gb300 as q
    c = _draw(case)
    wl = small_paged(c["seed"], num_seqs=c["seqs"], max_blocks=c["max_blocks"], block_size=c["bs"], rows=c["rows"],
                     topk=c["topk"], pad_frac=c["pad"], unallocated_frac=c["unalloc"],
                     num_q_heads=c["g"] * c["hkv"], num_kv_heads=c["hkv"], head_dim=c["hd"])
    R, Hq, D, P, K = wl.rows, wl.num_q_heads, wl.head_dim, c["P"], c["topk"]
    pos = wl.topk_pos.copy()
    lens = None
    if c["varlen"]:
        lens = np.random.default_rng(c["seed"]).integers(0, K + 1, R).astype(np.int32)
    slots, bad, _ = paged_slots(wl.block_table, wl.row_seq, pos, wl.block_size, wl.num_slots)
    ref_idx = slots.astype(np.int32)
    if lens is not None:
        for r in range(R):
            ref_idx[r, lens[r]:] = -1
            bad[r, lens[r]:] = False
            pos[r, lens[r]:] = 10 ** 8  # past a row's length: never read, never flagged
    wlr = dataclasses.replace(wl, topk=ref_idx)
    gp = GpuPool(wl, c["fmt"])
    out = torch.full((R, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((R, Hq), float("nan"), dtype=torch.float32, device="cuda")
    o_part = torch.empty((R, P, Hq, D), dtype=torch.float32, device="cuda") if P > 1 else None
    lse_part = torch.empty((R, P, Hq), dtype=torch.float32, device="cuda") if P > 1 else None
    counters = (torch.zeros((R, c["hkv"], (c["g"] + 15) // 16), dtype=torch.int32, device="cuda")
                if c["fused"] else None)
    sched = torch.zeros(2, dtype=torch.int32, device="cuda") if c["persistent"] else None
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = dict(num_kv_heads=c["hkv"], num_slots=wl.num_slots, k_scale_tok=gp.k_scale_tok, v_scale_tok=gp.v_scale_tok,
              k_scale_layer=float(gp.k_scale_layer), v_scale_layer=float(gp.v_scale_layer), dev_status=status,
              block_table=torch.from_numpy(np.ascontiguousarray(wl.block_table, dtype=np.int32)).cuda(),
              row_seq=torch.from_numpy(np.ascontiguousarray(wl.row_seq, dtype=np.int32)).cuda(),
              block_size=wl.block_size,
              topk_len=None if lens is None else torch.from_numpy(lens).cuda(),
              engine=q.QSA_ENGINE_PERSISTENT if c["persistent"] else q.QSA_ENGINE_DEFAULT, sched=sched)
    pos_dev = torch.from_numpy(np.ascontiguousarray(pos, dtype=np.int32)).cuda()
    if P == 1:
        q.qsa_gather_attn_ex(act_dev(wl.q), gp.code, gp.k_cache, gp.v_cache, pos_dev, wl.softmax_scale, out=out,
                             lse=lse, **kw)
    elif c["fused"]:
        q.qsa_gather_attn_ex(act_dev(wl.q), gp.code, gp.k_cache, gp.v_cache, pos_dev, wl.softmax_scale,
                             num_splits=P, out=out, lse=lse, o_part=o_part, lse_part=lse_part, counters=counters, **kw)
    else:
        q.qsa_gather_attn_ex(act_dev(wl.q), gp.code, gp.k_cache, gp.v_cache, pos_dev, wl.softmax_scale,
                             num_splits=P, o_part=o_part, lse_part=lse_part, **kw)
        q.qsa_splitk_merge(o_part, lse_part, out, lse,
                           v_scale_post=float(gp.v_scale_layer) if c["fmt"] == "e4m3" else 1.0)
    torch.cuda.synchronize()
    assert (status.item() == q.QKV_DEV_BAD_INDEX) == bool(bad.any()) and status.item() in (0, q.QKV_DEV_BAD_INDEX), c
    if counters is not None:
        assert int(counters.abs().sum().item()) == 0, c
    if sched is not None:
        assert sched.cpu().tolist() == [0, 0], c
    ro, rl = OraclePool(wlr, c["fmt"]).attend(wlr)
    assert_close(out.cpu().numpy(), ro, f"out {c}")
    assert_close(lse.cpu().numpy(), rl, f"lse {c}")

"""Very long rows against the fp64 oracle (GPU): top-k of tens of thousands per row.

A row then runs thousands of tiles per warp through one online softmax. Two of the rows are
ordered to stress that state:
- Ascending logits of head 0, so the running maximum keeps rising and the lazy rescale
  fires on tile after tile.
- Ascending V-token magnitude, so each new tile's largest V scale tends to exceed the bound
  in use, and the int8 V-scale bound is raised again and again.
Order does not change the attention itself (a row's keys are a set), so the oracle needs
nothing special. Checked unsplit, split with the separate merge, and split with the fused
merge; every output and lse element within |gpu - ref| <= 5e-5 + 1e-3 |ref|.
("int8 per-(token,head) KV cache for the Qwen3.8-Flash-Next QSA path" §The finding worth
upstreaming; "[Perf][SM70][FP8] Hoist QSA E4M3 KV scales" §Combined SM70 validation
provenance: long rows split over K.)
"""

import dataclasses

import numpy as np
import pytest
import torch

from gen import small_random
from harness import GpuPool, OraclePool, act_dev, assert_close

pytestmark = pytest.mark.gpu

TOPK = 48000


def _widen(bits):
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@pytest.fixture(scope="module")
def long_rows():
    wl = small_random(2027, num_slots=64000, num_tokens=60000, rows=3, topk=TOPK, outlier_frac=0.01,
                      pad_frac=0.02)
    idx = wl.topk.copy()
    tok_of_slot = np.full(wl.num_slots, -1, dtype=np.int64)
    tok_of_slot[wl.slot_mapping] = np.arange(wl.slot_mapping.size)
    k = _widen(wl.k_tokens[:, 0, :])  # [T, D] fp32, one KV head
    v = _widen(wl.v_tokens[:, 0, :])
    q0 = _widen(wl.q[0, 0, :])
    for r, key in ((0, lambda t: k[t] @ q0), (1, lambda t: np.abs(v[t]).max(axis=-1))):
        row = idx[r]
        valid = row >= 0
        toks = tok_of_slot[row[valid]]
        order = np.argsort(key(toks), kind="stable")
        idx[r] = np.concatenate([row[valid][order], row[~valid]])
    return dataclasses.replace(wl, topk=idx)


@pytest.mark.parametrize("fmt", ["int8_side", "int8_inline", "e4m3", "bf16"])
def test_long_rows_unsplit_and_split(long_rows, fmt):
    import quantized_kv_cache_write_gb300 as q
    wl = long_rows
    gp = GpuPool(wl, fmt)
    ro, rl = OraclePool(wl, fmt).attend(wl)
    out, lse, _, _ = gp.attend(wl)
    assert_close(out, ro, f"{fmt} unsplit out")
    assert_close(lse, rl, f"{fmt} unsplit lse")
    out, lse, _, _ = gp.attend(wl, num_splits=7)
    assert_close(out, ro, f"{fmt} split out")
    assert_close(lse, rl, f"{fmt} split lse")
    # fused merge: the last split CTA of each row merges; the counters come back zero
    R, Hq, D, P = wl.rows, wl.num_q_heads, wl.head_dim, 7
    o_part = torch.empty((R, P, Hq, D), dtype=torch.float32, device="cuda")
    lse_part = torch.empty((R, P, Hq), dtype=torch.float32, device="cuda")
    fo = torch.full((R, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    fl = torch.full((R, Hq), float("nan"), dtype=torch.float32, device="cuda")
    counters = torch.zeros((R, 1, 1), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = torch.from_numpy(np.ascontiguousarray(wl.topk, dtype=np.int32)).cuda()
    q.qsa_gather_attn_ex(act_dev(wl.q), gp.code, gp.k_cache, gp.v_cache, idx, wl.softmax_scale, num_slots=wl.num_slots,
                         k_scale_tok=gp.k_scale_tok, v_scale_tok=gp.v_scale_tok,
                         k_scale_layer=float(gp.k_scale_layer), v_scale_layer=float(gp.v_scale_layer),
                         num_splits=P, out=fo, lse=fl, o_part=o_part, lse_part=lse_part, counters=counters,
                         dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert int(counters.abs().sum().item()) == 0
    assert_close(fo.cpu().numpy(), ro, f"{fmt} fused out")
    assert_close(fl.cpu().numpy(), rl, f"{fmt} fused lse")

"""head_dim 128 on the GPU against the oracle.

The pages' model stores 256-wide heads ("int8 per-(token,head) KV cache for the
Qwen3.8-Flash-Next QSA path" §The finding worth upstreaming: 256 B of int8 data per head);
every entry point also takes 128-wide heads. Same bars as for 256: stored bytes bit-exact,
attention within |gpu - ref| <= 5e-5 + 1e-3 |ref| of the fp64 oracle, the fused and paged
paths bit-identical to the plain split path on the same slots.
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
D = 128


def _wl(seed, act="bf16", **kw):
    base = dict(num_slots=3000, rows=5, topk=333, pad_frac=0.05, outlier_frac=0.02, act_dtype=act, head_dim=D)
    base.update(kw)
    return small_random(seed, **base)


@pytest.mark.parametrize("act", ["bf16", "f16"])
@pytest.mark.parametrize("fmt", ["int8_side", "int8_inline", "e4m3"])
@pytest.mark.parametrize("large", [False, True])
def test_writes_are_bit_exact(fmt, act, large):
    """large: 18000 tokens, past the size where each warp writes a token's K and V rows."""
    wl = _wl(101, act, zero_tokens=2, **(dict(num_slots=20000, num_tokens=18000) if large else {}))
    gp, op = GpuPool(wl, fmt), OraclePool(wl, fmt)
    got = (gp.k_cache, gp.v_cache, gp.k_scale_tok, gp.v_scale_tok) if fmt == "int8_side" else (gp.k_cache, gp.v_cache)
    for g, r in zip(got, op.bytes):
        assert g.cpu().numpy().tobytes() == np.ascontiguousarray(r).tobytes()


@pytest.mark.parametrize("fmt,act", [("int8_side", "bf16"), ("int8_inline", "bf16"), ("e4m3", "bf16"),
                                     ("bf16", "bf16"), ("int8_side", "f16"), ("e4m3", "f16"), ("f16", "f16")])
@pytest.mark.parametrize("P", [1, 3])
def test_gather_matches_oracle(fmt, act, P):
    wl = _wl(102, act)
    wl.topk[2] = -1
    gp, op = GpuPool(wl, fmt), OraclePool(wl, fmt)
    out, lse, o_part, lse_part = gp.attend(wl, num_splits=P)
    ro, rl = op.attend(wl)
    assert_close(out, ro, f"{fmt} out")
    assert_close(lse, rl, f"{fmt} lse")
    assert np.all(out[2] == 0) and np.all(lse[2] == -np.inf)
    if P > 1:
        po, pl = op.attend_splits(wl, P)
        assert_close(o_part, po, f"{fmt} o_part")
        assert_close(lse_part, pl, f"{fmt} lse_part")


@pytest.mark.parametrize("fmt", ["int8_side", "e4m3", "bf16"])
def test_outlier_sweep_and_gqa32(fmt):
    for seed in range(6):
        wl = _wl(110 + seed, topk=64 + 150 * seed, outlier_frac=0.02 + 0.005 * seed,
                 num_q_heads=32 if seed % 3 == 2 else 16)
        out, lse, _, _ = GpuPool(wl, fmt).attend(wl)
        ro, rl = OraclePool(wl, fmt).attend(wl)
        assert_close(out, ro, f"{fmt} out seed {seed}")
        assert_close(lse, rl, f"{fmt} lse seed {seed}")


def test_fused_merge_is_bit_identical_and_counters_return_to_zero():
    import quantized_kv_cache_write_gb300 as q
    wl = _wl(103)
    gp = GpuPool(wl, "int8_side")
    R, Hq, P = wl.rows, wl.num_q_heads, 5
    out = torch.empty((R, Hq, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
    o_part = torch.empty((R, P, Hq, D), dtype=torch.float32, device="cuda")
    lse_part = torch.empty((R, P, Hq), dtype=torch.float32, device="cuda")
    counters = torch.zeros((R, 1, 1), dtype=torch.int32, device="cuda")
    idx = torch.from_numpy(wl.topk).cuda()
    q.qsa_gather_attn_splitk_fused(act_dev(wl.q), gp.code, gp.k_cache, gp.v_cache, idx, wl.softmax_scale,
                                   num_splits=P, out=out, lse=lse, o_part=o_part, lse_part=lse_part,
                                   counters=counters, k_scale_tok=gp.k_scale_tok, v_scale_tok=gp.v_scale_tok)
    torch.cuda.synchronize()
    ref = gp.attend(wl, num_splits=P)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref[0].view(np.uint32))
    assert np.array_equal(lse.cpu().numpy().view(np.uint32), ref[1].view(np.uint32))
    assert int(counters.abs().sum().item()) == 0


def test_noalloc_matches_the_plain_split_path():
    import quantized_kv_cache_write_gb300 as q
    wl = _wl(104)
    gp = GpuPool(wl, "e4m3")
    out = torch.empty((wl.rows, wl.num_q_heads, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((wl.rows, wl.num_q_heads), dtype=torch.float32, device="cuda")
    q.qsa_gather_attn_splitk_noalloc(act_dev(wl.q), gp.code, gp.k_cache, gp.v_cache,
                                     torch.from_numpy(wl.topk).cuda(), wl.softmax_scale, num_splits=4, out=out,
                                     lse=lse, k_scale_layer=float(gp.k_scale_layer),
                                     v_scale_layer=float(gp.v_scale_layer))
    torch.cuda.synchronize()
    ref = gp.attend(wl, num_splits=4)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref[0].view(np.uint32))


@pytest.mark.parametrize("fmt", ["int8_side", "bf16"])
def test_paged_pool(fmt):
    import quantized_kv_cache_write_gb300 as q
    wl = small_paged(105, head_dim=D)
    slots, bad, bad_row = paged_slots(wl.block_table, wl.row_seq, wl.topk_pos, wl.block_size, wl.num_slots)
    wls = dataclasses.replace(wl, topk=slots.astype(np.int32))
    gp = GpuPool(wls, fmt)
    out = torch.empty((wl.rows, wl.num_q_heads, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((wl.rows, wl.num_q_heads), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q.qsa_gather_attn_paged(act_dev(wl.q), gp.code, gp.k_cache, gp.v_cache,
                            torch.from_numpy(wl.block_table).cuda(), torch.from_numpy(wl.row_seq).cuda(),
                            torch.from_numpy(wl.topk_pos).cuda(), wl.block_size, wl.softmax_scale, out=out, lse=lse,
                            k_scale_tok=gp.k_scale_tok, v_scale_tok=gp.v_scale_tok, dev_status=status)
    torch.cuda.synchronize()
    ro, rl = OraclePool(wls, fmt).attend(wls)
    assert_close(out.cpu().numpy(), ro, "paged out")
    assert_close(lse.cpu().numpy(), rl, "paged lse")
    assert (status.item() != 0) == bool(bad.any() or bad_row.any())


def test_merge_kernel():
    import quantized_kv_cache_write_gb300 as q
    rng = np.random.default_rng(106)
    R, P, Hq = 5, 7, 16
    op = rng.standard_normal((R, P, Hq, D)).astype(np.float32)
    lp = (rng.standard_normal((R, P, Hq)) * 5).astype(np.float32)
    lp[rng.random((R, P, Hq)) < 0.2] = -np.inf
    lp[1] = -np.inf
    out = torch.empty((R, Hq, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
    q.qsa_splitk_merge(torch.from_numpy(op).cuda(), torch.from_numpy(lp).cuda(), out, lse, v_scale_post=0.5)
    ro, rl = oatt.merge_splits(op.astype(np.float64), lp.astype(np.float64), v_scale_post=0.5)
    assert_close(out.cpu().numpy(), ro, "merge out", atol=1e-6, rtol=1e-5)
    assert_close(lse.cpu().numpy(), rl, "merge lse", atol=1e-6, rtol=1e-5)

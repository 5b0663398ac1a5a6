"""qsa_gather_attn_varlen: rows of different lengths (GPU).

Row r uses topk_idx[r, :topk_len[r]]; the entries past its length are never read, so they may
hold anything (here: out-of-range garbage that would be flagged if read). The result must
equal the oracle on the same rows with those entries set to -1 padding. Batches that mix
long and short rows are what the calibrated E4M3 page routes across kernels
("[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache" §Implementation scope).
"""

import numpy as np
import pytest
import torch

from gen import chunked_prefill, small_random
from harness import GpuPool, OraclePool, act_dev, assert_close
from oracle import attention as oatt

pytestmark = pytest.mark.gpu
FORMATS = ["int8_side", "int8_inline", "e4m3", "bf16"]


def _run(gp, wl, idx, lens, P, status=None):
    import quantized_kv_cache_write_gb300 as q
    R, Hq, D = wl.rows, wl.num_q_heads, wl.head_dim
    out = torch.full((R, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((R, Hq), float("nan"), dtype=torch.float32, device="cuda")
    kw = dict(k_scale_tok=gp.k_scale_tok, v_scale_tok=gp.v_scale_tok, k_scale_layer=float(gp.k_scale_layer),
              v_scale_layer=float(gp.v_scale_layer), num_kv_heads=wl.num_kv_heads, num_slots=wl.num_slots,
              dev_status=status)
    idx_d = torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).cuda()
    len_d = torch.from_numpy(np.ascontiguousarray(lens, dtype=np.int32)).cuda()
    if P == 1:
        q.qsa_gather_attn_varlen(act_dev(wl.q), gp.code, gp.k_cache, gp.v_cache, idx_d, len_d, wl.softmax_scale,
                                 out=out, lse=lse, **kw)
    else:
        o_part = torch.empty((R, P, Hq, D), dtype=torch.float32, device="cuda")
        lse_part = torch.empty((R, P, Hq), dtype=torch.float32, device="cuda")
        q.qsa_gather_attn_varlen(act_dev(wl.q), gp.code, gp.k_cache, gp.v_cache, idx_d, len_d, wl.softmax_scale,
                                 num_splits=P, o_part=o_part, lse_part=lse_part, **kw)
        q.qsa_splitk_merge(o_part, lse_part, out, lse,
                           v_scale_post=float(gp.v_scale_layer) if gp.fmt == "e4m3" else 1.0)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("P", [1, 4])
def test_rows_of_different_lengths(fmt, P):
    wl = small_random(131, num_slots=4000, rows=9, topk=600, pad_frac=0.05, outlier_frac=0.01)
    rng = np.random.default_rng(7)
    lens = rng.integers(0, 601, wl.rows)
    lens[0], lens[1], lens[2] = 0, 600, 1
    idx = wl.topk.copy()
    garbage = idx.copy()
    for r in range(wl.rows):
        garbage[r, lens[r]:] = rng.integers(10 ** 6, 10 ** 9, wl.topk.shape[1] - lens[r])  # never read
        idx[r, lens[r]:] = -1
    gp = GpuPool(wl, fmt)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = _run(gp, wl, garbage, lens, P, status)
    assert status.item() == 0  # nothing past a row's length was read
    op = OraclePool(wl, fmt)
    ro, rl = oatt.gather_attention(wl.q, op.K, op.V, idx, wl.softmax_scale)
    assert_close(out, ro, f"{fmt} out")
    assert_close(lse, rl, f"{fmt} lse")
    assert np.all(out[0] == 0) and np.all(lse[0] == -np.inf)


def test_lengths_outside_the_width_are_flagged_and_clamped():
    wl = small_random(132, num_slots=2000, rows=3, topk=50)
    gp = GpuPool(wl, "int8_side")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = _run(gp, wl, wl.topk, np.array([-3, 50, 77]), 1, status)
    assert status.item() == 2
    idx = wl.topk.copy()
    idx[0] = -1
    op = OraclePool(wl, "int8_side")
    ro, rl = oatt.gather_attention(wl.q, op.K, op.V, idx, wl.softmax_scale)
    assert_close(out, ro, "out")
    assert_close(lse, rl, "lse")


def test_chunked_prefill_rows_by_length():
    wl = chunked_prefill(4)
    lens = np.minimum(np.arange(wl.rows), wl.topk.shape[1])
    gp = GpuPool(wl, "int8_side")
    out, lse = _run(gp, wl, wl.topk, lens, 1)
    rows = np.array([0, 1, 2, 63, 64, 1000, 1023, 1024, 1025, 4096, 8191])
    ro, rl = OraclePool(wl, "int8_side").attend(wl, rows=rows)
    assert_close(out[rows], ro[rows], "out")
    assert_close(lse[rows], rl[rows], "lse")

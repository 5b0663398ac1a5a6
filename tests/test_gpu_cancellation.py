"""Near cancellations of two outlier keys against the fp64 oracle (GPU).

Each row's output is the small difference of two large terms: a pair of outlier keys with
equal or nearly equal K and exactly opposite V sits 8 or 40 above the row's other logits
(gen.cancelling_pairs). Outputs are ~1e-3 of the terms they cancel (|V| up to ~60). There the
stated tolerance, 5e-5 + 1e-3 |ref|, asks for ~1e-6 of the cancelled magnitude, which no fp32
pipeline guarantees: attention in plain fp32 misses it on this fixture
(tests/test_gen.py::test_cancelling_pairs_exceed_fp32_precision), and so do the kernels on
some seeds (bf16 by up to 3x, E4M3 by up to 2x, int8 by up to 1.25x). So outputs are checked
against the tolerance plus 2^-16 of the magnitude being cancelled, m = sum p |V| / sum p (the
oracle's own attention with |V|): the truncation of up to ~128 fp32 tensor-core accumulation
steps on terms of size m. A dropped p_lo part (2^-12 m) or a logit off by 1e-4 fails it.
lse is not cancelled and keeps the plain tolerance. Every pool layout, unsplit and split;
the int8 side layout also through the tcgen05 and persistent engines.
("int8 per-(token,head) KV cache for the Qwen3.8-Flash-Next QSA path" §The finding worth
upstreaming: outlier tokens are what the per-(token, head) scale is for.)
"""

import numpy as np
import pytest
import torch

from gen import cancelling_pairs
from harness import ATOL, GpuPool, OraclePool, act_dev, assert_close
from oracle import attention as oatt

pytestmark = pytest.mark.gpu

COND = 2.0 ** -16  # of the cancelled magnitude m


@pytest.fixture(scope="module")
def wl():
    return cancelling_pairs()


def _ref_and_allowance(wl, fmt):
    op = OraclePool(wl, fmt)
    ro, rl = op.attend(wl)
    m, _ = oatt.gather_attention(wl.q, op.K, np.abs(op.V), wl.topk, wl.softmax_scale)
    return ro, rl, ATOL + COND * m


@pytest.mark.parametrize("fmt", ["int8_side", "int8_inline", "e4m3", "bf16"])
def test_near_cancellation_unsplit_and_split(wl, fmt):
    gp = GpuPool(wl, fmt)
    ro, rl, atol = _ref_and_allowance(wl, fmt)
    for P in (1, 3):
        out, lse, _, _ = gp.attend(wl, num_splits=P)
        assert_close(out, ro, f"{fmt} P={P} out", atol=atol)
        assert_close(lse, rl, f"{fmt} P={P} lse")


@pytest.mark.parametrize("engine", ["tcgen05", "persistent"])
def test_near_cancellation_other_engines(wl, engine):
    import quantized_kv_cache_write_gb300 as q
    gp = GpuPool(wl, "int8_side")
    ro, rl, atol = _ref_and_allowance(wl, "int8_side")
    R, Hq, D = wl.rows, wl.num_q_heads, wl.head_dim
    out = torch.full((R, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((R, Hq), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sched = torch.zeros(2, dtype=torch.int32, device="cuda") if engine == "persistent" else None
    code = q.QSA_ENGINE_TCGEN05 if engine == "tcgen05" else q.QSA_ENGINE_PERSISTENT
    idx = torch.from_numpy(np.ascontiguousarray(wl.topk, dtype=np.int32)).cuda()
    q.qsa_gather_attn_ex(act_dev(wl.q), gp.code, gp.k_cache, gp.v_cache, idx, wl.softmax_scale,
                         num_slots=wl.num_slots, k_scale_tok=gp.k_scale_tok, v_scale_tok=gp.v_scale_tok,
                         out=out, lse=lse, dev_status=status, engine=code, sched=sched)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert_close(out.cpu().numpy(), ro, f"{engine} out", atol=atol)
    assert_close(lse.cpu().numpy(), rl, f"{engine} lse")


@pytest.mark.parametrize("seed", [9, 10, 11, 12, 13])
def test_near_cancellation_more_seeds(seed):
    w = cancelling_pairs(seed=seed)
    for fmt in ("int8_side", "e4m3", "bf16"):
        gp = GpuPool(w, fmt)
        ro, rl, atol = _ref_and_allowance(w, fmt)
        out, lse, _, _ = gp.attend(w)
        assert_close(out, ro, f"seed {seed} {fmt} out", atol=atol)
        assert_close(lse, rl, f"seed {seed} {fmt} lse")

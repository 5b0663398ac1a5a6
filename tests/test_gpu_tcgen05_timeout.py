"""The tcgen05 engine's lost-wait path, made to run out on purpose (GPU).

The engine's warps hand blocks to each other through mbarriers, and every wait is bounded: one
that runs out sets QKV_DEV_TIMEOUT and the CTA winds down (its own copies and MMAs drained, its
tensor memory freed). QKV_TEST_TCGEN05_DROP_HANDOFF=<block> makes the compute warps leave out
one block's K hand-off to the MMA warp, a wait that nothing will satisfy: the MMA warp's wait
for it and the compute warps' wait for that block's scores run out (after 2^14 polls in this
mode). Nothing faults and nothing hangs. The launch must come back with the timeout bit set,
and the same context must then run the engine normally and match the oracle.
"""

import os

import numpy as np
import pytest
import torch

from gen import small_random
from harness import GpuPool, OraclePool, act_dev, assert_close

pytestmark = pytest.mark.gpu

ENV = "QKV_TEST_TCGEN05_DROP_HANDOFF"


def _launch(q, wl, gp, out, lse, status):
    idx = torch.from_numpy(np.ascontiguousarray(wl.topk, dtype=np.int32)).cuda()
    q.qsa_gather_attn_ex(act_dev(wl.q), gp.code, gp.k_cache, gp.v_cache, idx, wl.softmax_scale, num_slots=wl.num_slots,
                         k_scale_tok=gp.k_scale_tok, v_scale_tok=gp.v_scale_tok, out=out, lse=lse, dev_status=status,
                         engine=q.QSA_ENGINE_TCGEN05)
    torch.cuda.synchronize()


@pytest.mark.parametrize("block", [0, 1, 5])
def test_a_lost_handoff_times_out_and_the_context_stays_usable(block):
    import quantized_kv_cache_write_gb300 as q
    assert ENV not in os.environ
    wl = small_random(71, num_slots=8000, rows=12, topk=900, pad_frac=0.05, outlier_frac=0.02)
    gp = GpuPool(wl, "int8_side")
    R, Hq, D = wl.rows, wl.num_q_heads, wl.head_dim
    out = torch.empty((R, Hq, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    os.environ[ENV] = str(block)
    try:
        _launch(q, wl, gp, out, lse, status)
    finally:
        del os.environ[ENV]
    assert status.item() & q.QKV_DEV_TIMEOUT, status.item()
    # the same context, the same buffers: a normal launch is clean and correct
    status.zero_()
    out.fill_(float("nan"))
    _launch(q, wl, gp, out, lse, status)
    assert status.item() == 0
    ro, rl = OraclePool(wl, "int8_side").attend(wl)
    assert_close(out.cpu().numpy(), ro, "out after the timeout")
    assert_close(lse.cpu().numpy(), rl, "lse after the timeout")

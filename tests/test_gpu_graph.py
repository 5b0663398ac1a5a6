"""The library under CUDA-graph capture (GPU).

"[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache" §Validation runs the decode step as a
captured CUDA graph (FULL_AND_PIECEWISE). The library enqueues only kernel launches on the
caller's stream, with no allocation or synchronisation, so a decode step -- quantize-on-write
of the new tokens, then the gather with its fused split-K merge -- can be captured once and
replayed. Replays must give the eager results bit for bit and leave the arrival counters at
zero.
"""

import numpy as np
import pytest
import torch

from gen import small_random
from harness import GpuPool, act_dev

pytestmark = pytest.mark.gpu


def test_captured_decode_step_replays_bit_exactly():
    import quantized_kv_cache_write_gb300 as q
    wl = small_random(121, num_slots=5000, rows=8, topk=700, num_tokens=4000, pad_frac=0.05, outlier_frac=0.01)
    gp = GpuPool(wl, "int8_side")
    rng = np.random.default_rng(5)
    T = 16  # this step's new tokens go to slots no row reads
    free = np.setdiff1d(np.arange(wl.num_slots), wl.slot_mapping)
    new_slots = torch.from_numpy(rng.choice(free, T, replace=False).astype(np.int64)).cuda()
    new_k = torch.randn((T, 1, 256), device="cuda").to(torch.bfloat16)
    new_v = torch.randn((T, 1, 256), device="cuda").to(torch.bfloat16)
    qd = act_dev(wl.q)
    idx = torch.from_numpy(wl.topk).cuda()
    R, Hq, D, P = wl.rows, wl.num_q_heads, 256, 6
    out = torch.empty((R, Hq, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
    o_part = torch.empty((R, P, Hq, D), dtype=torch.float32, device="cuda")
    lse_part = torch.empty((R, P, Hq), dtype=torch.float32, device="cuda")
    counters = torch.zeros((R, 1, 1), dtype=torch.int32, device="cuda")

    def step():
        q.qkv_write_int8(new_k, new_v, new_slots, gp.k_cache, gp.v_cache, gp.k_scale_tok, gp.v_scale_tok)
        q.qsa_gather_attn_splitk_fused(qd, gp.code, gp.k_cache, gp.v_cache, idx, wl.softmax_scale, num_splits=P,
                                       out=out, lse=lse, o_part=o_part, lse_part=lse_part, counters=counters,
                                       k_scale_tok=gp.k_scale_tok, v_scale_tok=gp.v_scale_tok)

    step()  # eager: the first call on a device also sets the kernels' attributes
    torch.cuda.synchronize()
    ref_out, ref_lse = out.clone(), lse.clone()
    ref_k = gp.k_cache.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up on the capture stream, as torch recommends before capturing
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int32), ref_out.view(torch.int32))
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))
        assert torch.equal(gp.k_cache, ref_k)
        assert int(counters.abs().sum().item()) == 0

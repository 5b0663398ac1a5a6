"""Seeded random configurations of the gather against the fp64 oracle (GPU).

Each case draws a pool layout, head dim, GQA group, KV-head count, row count, top-k width,
padding and outlier fractions, per-row lengths (or none), a split count, the fused merge (or
the separate merge), an engine and the query type (bf16, or fp16 with fp16 tokens written
into the pool), then checks every output and lse element within
|gpu - ref| <= 5e-5 + 1e-3 |ref| and that nothing was flagged. The draws are seeded, so a
failure names a reproducible configuration.
"""

import dataclasses

import numpy as np
import pytest
import torch

from gen import small_random
from harness import GpuPool, OraclePool, act_dev, assert_close

pytestmark = pytest.mark.gpu

FORMATS = ["int8_side", "int8_inline", "e4m3", "bf16", "f16"]


def _draw(seed):
    rng = np.random.default_rng([20251202, seed])
    fmt = FORMATS[rng.integers(len(FORMATS))]
    hd = int(rng.choice([128, 256]))
    hkv = int(rng.choice([1, 1, 2]))
    g = int(rng.choice([1, 3, 8, 16, 16, 20, 32]))
    rows = int(rng.integers(1, 24))
    topk = int(rng.choice([1, 15, 16, 17, 100, 257, 700, 1500]))
    P = int(rng.choice([1, 1, 2, 3, 8]))
    fused = bool(rng.integers(2)) and P > 1
    varlen = bool(rng.integers(2))
    pad = float(rng.choice([0.0, 0.0, 0.2]))
    outl = float(rng.choice([0.0, 0.02, 0.05]))
    engine = "default"
    if rng.integers(3) == 0:
        engine = "persistent"
    elif fmt == "int8_side" and hd == 256 and g <= 16 and not fused and rng.integers(3) == 0:
        engine = "tcgen05"
    seed = int(rng.integers(1 << 30))
    # the query type, drawn last so that the draws above stay as they were: an unquantised pool
    # takes a query of its own type; int8 and E4M3 pools take either (the FP16-activation
    # contract), except on the tcgen05 engine (bf16 queries only)
    act = "f16" if fmt == "f16" else "bf16"
    if fmt in ("int8_side", "int8_inline", "e4m3") and engine != "tcgen05" and rng.integers(3) == 0:
        act = "f16"
    return dict(fmt=fmt, hd=hd, hkv=hkv, g=g, rows=rows, topk=topk, P=P, fused=fused, varlen=varlen, pad=pad,
                outl=outl, engine=engine, seed=seed, act=act)


@pytest.mark.parametrize("case", range(96))
def test_random_configuration(case):
    import quantized_kv_cache_write_gb300 as q
    c = _draw(case)
    act = c["act"]
    wl = small_random(c["seed"], num_slots=3000, rows=c["rows"], topk=c["topk"], num_q_heads=c["g"] * c["hkv"],
                      num_kv_heads=c["hkv"], pad_frac=c["pad"], outlier_frac=c["outl"], act_dtype=act,
                      head_dim=c["hd"])
    idx = wl.topk.copy()
    lens = None
    if c["varlen"]:
        rng = np.random.default_rng(c["seed"])
        lens = rng.integers(0, c["topk"] + 1, c["rows"]).astype(np.int32)
        for r in range(c["rows"]):
            idx[r, lens[r]:] = -1
    wlc = wl if lens is None else dataclasses.replace(wl, topk=idx)
    gp = GpuPool(wlc, c["fmt"])
    R, Hq, D, P = c["rows"], wl.num_q_heads, c["hd"], c["P"]
    out = torch.full((R, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((R, Hq), float("nan"), dtype=torch.float32, device="cuda")
    o_part = torch.empty((R, P, Hq, D), dtype=torch.float32, device="cuda") if P > 1 else None
    lse_part = torch.empty((R, P, Hq), dtype=torch.float32, device="cuda") if P > 1 else None
    counters = (torch.zeros((R, c["hkv"], (c["g"] + 15) // 16), dtype=torch.int32, device="cuda")
                if c["fused"] else None)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    engine = {"default": q.QSA_ENGINE_DEFAULT, "persistent": q.QSA_ENGINE_PERSISTENT,
              "tcgen05": q.QSA_ENGINE_TCGEN05}[c["engine"]]
    sched = torch.zeros(2, dtype=torch.int32, device="cuda") if c["engine"] == "persistent" else None
    kw = dict(num_kv_heads=c["hkv"], num_slots=wl.num_slots, k_scale_tok=gp.k_scale_tok, v_scale_tok=gp.v_scale_tok,
              k_scale_layer=float(gp.k_scale_layer), v_scale_layer=float(gp.v_scale_layer), dev_status=status,
              engine=engine, sched=sched,
              topk_len=None if lens is None else torch.from_numpy(lens).cuda())
    # entries past a row's length are never read: fill them with out-of-range garbage
    idx_dev = wl.topk.copy()
    if lens is not None:
        for r in range(R):
            idx_dev[r, lens[r]:] = 10 ** 8
    idx_dev = torch.from_numpy(np.ascontiguousarray(idx_dev, dtype=np.int32)).cuda()
    if P == 1:
        q.qsa_gather_attn_ex(act_dev(wl.q, act), gp.code, gp.k_cache, gp.v_cache, idx_dev, wl.softmax_scale,
                             out=out, lse=lse, **kw)
    elif c["fused"]:
        q.qsa_gather_attn_ex(act_dev(wl.q, act), gp.code, gp.k_cache, gp.v_cache, idx_dev, wl.softmax_scale,
                             num_splits=P, out=out, lse=lse, o_part=o_part, lse_part=lse_part, counters=counters,
                             **kw)
    else:
        q.qsa_gather_attn_ex(act_dev(wl.q, act), gp.code, gp.k_cache, gp.v_cache, idx_dev, wl.softmax_scale,
                             num_splits=P, o_part=o_part, lse_part=lse_part, **kw)
        q.qsa_splitk_merge(o_part, lse_part, out, lse,
                           v_scale_post=float(gp.v_scale_layer) if c["fmt"] == "e4m3" else 1.0)
    torch.cuda.synchronize()
    assert status.item() == 0, c
    if counters is not None:
        assert int(counters.abs().sum().item()) == 0, c
    if sched is not None:
        assert sched.cpu().tolist() == [0, 0], c
    ro, rl = OraclePool(wlc, c["fmt"]).attend(wlc)
    assert_close(out.cpu().numpy(), ro, f"out {c}")
    assert_close(lse.cpu().numpy(), rl, f"lse {c}")

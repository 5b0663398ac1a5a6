"""One named case of the library's kernels, launched a few times: the command a profiler wraps.

    python -m quantized_kv_cache_write_gb300.profile_cases <case> [--launches N]

Each case builds its slot pool with the library's own write kernels from the seeded
generator's inputs, then launches the case's gather N times (default 3), each after an L2
flush (a 256 MiB write), and synchronises. Profile the last launch with
`-k regex:<kernel> -s <N - 1> -c 1`. Cases:

  page1_<fmt>        2048 rows x top-k 1024 over 262144 slots, fmt = int8_side, int8_inline,
                     e4m3 or bf16 ("int8 per-(token,head) KV cache for the Qwen3.8-Flash-Next
                     QSA path", §The finding worth upstreaming)
  page1_tcgen05      the same, int8 side, QSA_ENGINE_TCGEN05
  page1_gqa32        the same, int8 side, 32 query heads on one KV head
  page1_hd128        the same, int8 side, head_dim 128 (128 B of codes per head row)
  e4m3_layer         one calibrated E4M3 layer: 64 rows x top-k 2051 over 131072 slots, fused
                     split-K at qsa_suggest_num_splits' count ("[Perf][SM70][FP8] Hoist QSA
                     E4M3 KV scales", §Combined SM70 validation provenance)
  long_context       40 rows x top-k 2048 of 8 x 131072-token sequences, int8 side, fused at
                     the suggested split count
  mixed_<engine>     the 49-row catch-up/decode batch, E4M3, varlen, fused, 8 splits, engine =
                     default or persistent ("[Model][SM70][FP8] Add calibrated E4M3 QSA KV
                     cache", §Targeted mixed-batch scheduler regression)
  chunked_prefill    8192 causal rows (row i attends min(1024, i) of the 8192 tokens just
                     written into a 524288-slot int8 side pool), varlen
  write_<fmt>_fill   the page-1 pool fill: 262144 bf16 tokens written into a 262144-slot pool,
                     fmt = int8 (side tensors) or e4m3 (calibrated scales)
  merge_e4m3_layer   qsa_splitk_merge of the E4M3 layer's split partials (64 rows, 16 heads, P
                     from qsa_suggest_num_splits), the separate-merge path
"""

from __future__ import annotations

import argparse
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import quantized_kv_cache_write_gb300 as q  # noqa: E402
from gen import (chunked_prefill, e4m3_splitk_layer, long_context_decode, mixed_catchup_decode,  # noqa: E402
                 page1_shape, small_random)

CASES = ["page1_int8_side", "page1_int8_inline", "page1_e4m3", "page1_bf16", "page1_tcgen05", "page1_gqa32",
         "page1_hd128", "e4m3_layer", "long_context", "mixed_default", "mixed_persistent", "chunked_prefill",
         "write_int8_fill", "write_e4m3_fill", "merge_e4m3_layer"]


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _pool(wl, fmt):
    """The workload's tokens written by the library: caches and the gather's scale arguments."""
    S, H, D = wl.num_slots, wl.num_kv_heads, wl.head_dim
    k, v, slots = _dev(wl.k_tokens), _dev(wl.v_tokens), torch.from_numpy(wl.slot_mapping).cuda()
    if fmt == "bf16":
        kc = torch.zeros((S, H, D), dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        kc[slots], vc[slots] = k, v
        return kc, vc, {}
    if fmt in ("int8_side", "int8_inline"):
        side = fmt == "int8_side"
        kc = torch.zeros((S, H, D if side else D + 4), dtype=torch.int8 if side else torch.uint8, device="cuda")
        vc = torch.zeros_like(kc)
        if side:
            ks = torch.zeros((S, H), dtype=torch.float32, device="cuda")
            vs = torch.zeros_like(ks)
            q.qkv_write_int8(k, v, slots, kc, vc, ks, vs)
            return kc, vc, dict(k_scale_tok=ks, v_scale_tok=vs)
        q.qkv_write_int8(k, v, slots, kc, vc, layout=q.QKV_INT8_INLINE)
        return kc, vc, {}
    amax = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc = torch.zeros(2, dtype=torch.float32, device="cuda")
    q.qkv_e4m3_calibrate(k, amax, sc[0:1])
    q.qkv_e4m3_calibrate(v, amax, sc[1:2])
    ksl, vsl = sc.tolist()
    kc = torch.zeros((S, H, D), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    q.qkv_write_e4m3(k, v, slots, kc, vc, ksl, vsl)
    return kc, vc, dict(k_scale_layer=ksl, v_scale_layer=vsl)


def build(case: str):
    """The case's launch as a closure (inputs resident on the device)."""
    if case.startswith("page1_"):
        what = case[len("page1_"):]
        if what == "gqa32":
            wl, fmt = small_random(11, num_slots=262144, rows=2048, topk=1024, outlier_frac=0.01, num_q_heads=32), \
                "int8_side"
        elif what == "hd128":
            wl, fmt = small_random(11, num_slots=262144, rows=2048, topk=1024, outlier_frac=0.01, head_dim=128), \
                "int8_side"
        else:
            wl, fmt = page1_shape(1, with_step=False), ("int8_side" if what == "tcgen05" else what)
        kc, vc, kw = _pool(wl, fmt)
        qd, idx = _dev(wl.q), torch.from_numpy(np.ascontiguousarray(wl.topk, dtype=np.int32)).cuda()
        out = torch.empty((wl.rows, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device="cuda")
        engine = q.QSA_ENGINE_TCGEN05 if what == "tcgen05" else q.QSA_ENGINE_DEFAULT
        return lambda: q.qsa_gather_attn_ex(qd, q.FORMATS[fmt], kc, vc, idx, wl.softmax_scale, out=out,
                                            engine=engine, **kw)
    if case in ("e4m3_layer", "long_context"):
        wl, fmt = (e4m3_splitk_layer(0), "e4m3") if case == "e4m3_layer" else (long_context_decode(3), "int8_side")
        kc, vc, kw = _pool(wl, fmt)
        qd, idx = _dev(wl.q), torch.from_numpy(np.ascontiguousarray(wl.topk, dtype=np.int32)).cuda()
        R, Hq, D = wl.rows, wl.num_q_heads, wl.head_dim
        P = q.qsa_suggest_num_splits(q.FORMATS[fmt], R, Hq, wl.num_kv_heads, wl.topk.shape[1])
        out = torch.empty((R, Hq, D), dtype=torch.float32, device="cuda")
        o_part = torch.empty((R, P, Hq, D), dtype=torch.float32, device="cuda")
        lse_part = torch.empty((R, P, Hq), dtype=torch.float32, device="cuda")
        counters = torch.zeros((R, wl.num_kv_heads, 1), dtype=torch.int32, device="cuda")
        return lambda: q.qsa_gather_attn_splitk_fused(qd, q.FORMATS[fmt], kc, vc, idx, wl.softmax_scale, num_splits=P,
                                                      out=out, o_part=o_part, lse_part=lse_part, counters=counters,
                                                      **kw)
    if case in ("mixed_default", "mixed_persistent"):
        wl = mixed_catchup_decode(6)
        kc, vc, kw = _pool(wl, "e4m3")
        qd, idx = _dev(wl.q), torch.from_numpy(np.ascontiguousarray(wl.topk, dtype=np.int32)).cuda()
        lens = torch.from_numpy(wl.row_len).cuda()
        R, Hq, D, P = wl.rows, wl.num_q_heads, wl.head_dim, wl.num_splits
        out = torch.empty((R, Hq, D), dtype=torch.float32, device="cuda")
        o_part = torch.empty((R, P, Hq, D), dtype=torch.float32, device="cuda")
        lse_part = torch.empty((R, P, Hq), dtype=torch.float32, device="cuda")
        counters = torch.zeros((R, 1, 1), dtype=torch.int32, device="cuda")
        sched = torch.zeros(2, dtype=torch.int32, device="cuda")
        engine = q.QSA_ENGINE_PERSISTENT if case == "mixed_persistent" else q.QSA_ENGINE_DEFAULT
        return lambda: q.qsa_gather_attn_ex(qd, q.QKV_E4M3, kc, vc, idx, wl.softmax_scale, num_splits=P, out=out,
                                            o_part=o_part, lse_part=lse_part, counters=counters, topk_len=lens,
                                            engine=engine, sched=sched if engine == q.QSA_ENGINE_PERSISTENT else None,
                                            **kw)
    if case == "chunked_prefill":
        wl = chunked_prefill(4)
        kc, vc, kw = _pool(wl, "int8_side")
        qd, idx = _dev(wl.q), torch.from_numpy(np.ascontiguousarray(wl.topk, dtype=np.int32)).cuda()
        lens = torch.from_numpy(np.minimum(np.arange(wl.rows), wl.topk.shape[1]).astype(np.int32)).cuda()
        out = torch.empty((wl.rows, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device="cuda")
        return lambda: q.qsa_gather_attn_varlen(qd, q.QKV_INT8_SIDE, kc, vc, idx, lens, wl.softmax_scale, out=out,
                                                **kw)
    if case in ("write_int8_fill", "write_e4m3_fill"):
        wl = page1_shape(1, with_step=False)
        S, H, D = wl.num_slots, wl.num_kv_heads, wl.head_dim
        k, v, slots = _dev(wl.k_tokens), _dev(wl.v_tokens), torch.from_numpy(wl.slot_mapping).cuda()
        kc = torch.zeros((S, H, D), dtype=torch.int8 if case == "write_int8_fill" else torch.uint8, device="cuda")
        vc = torch.zeros_like(kc)
        if case == "write_int8_fill":
            ks = torch.zeros((S, H), dtype=torch.float32, device="cuda")
            vs = torch.zeros_like(ks)
            return lambda: q.qkv_write_int8(k, v, slots, kc, vc, ks, vs)
        amax = torch.zeros(1, dtype=torch.int32, device="cuda")
        sc = torch.zeros(2, dtype=torch.float32, device="cuda")
        q.qkv_e4m3_calibrate(k, amax, sc[0:1])
        q.qkv_e4m3_calibrate(v, amax, sc[1:2])
        ksl, vsl = sc.tolist()
        return lambda: q.qkv_write_e4m3(k, v, slots, kc, vc, ksl, vsl)
    if case == "merge_e4m3_layer":
        wl = e4m3_splitk_layer(0)
        kc, vc, kw = _pool(wl, "e4m3")
        qd, idx = _dev(wl.q), torch.from_numpy(np.ascontiguousarray(wl.topk, dtype=np.int32)).cuda()
        R, Hq, D = wl.rows, wl.num_q_heads, wl.head_dim
        P = q.qsa_suggest_num_splits(q.QKV_E4M3, R, Hq, wl.num_kv_heads, wl.topk.shape[1])
        o_part = torch.empty((R, P, Hq, D), dtype=torch.float32, device="cuda")
        lse_part = torch.empty((R, P, Hq), dtype=torch.float32, device="cuda")
        q.qsa_gather_attn(qd, q.QKV_E4M3, kc, vc, idx, wl.softmax_scale, num_splits=P, o_part=o_part,
                          lse_part=lse_part, **kw)
        out = torch.empty((R, Hq, D), dtype=torch.float32, device="cuda")
        lse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
        return lambda: q.qsa_splitk_merge(o_part, lse_part, out, lse, v_scale_post=float(kw["v_scale_layer"]))
    raise SystemExit(f"unknown case {case!r}; one of {', '.join(CASES)}")


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("case", choices=CASES)
    ap.add_argument("--launches", type=int, default=3)
    args = ap.parse_args()
    if not torch.cuda.is_available():
        raise SystemExit("profile_cases needs a CUDA device")
    run = build(args.case)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for i in range(args.launches):
        flush.fill_(i & 0xFF)
        run()
    torch.cuda.synchronize()
    print(f"{args.case}: {args.launches} launches done")


if __name__ == "__main__":
    main()

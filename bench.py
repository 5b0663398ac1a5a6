#!/usr/bin/env python3
"""Benchmark of one decode step of the quantized-KV top-k gather path on GB300.

Workload (the page-1 micro-benchmark shape of "int8 per-(token,head) KV cache for the
Qwen3.8-Flash-Next QSA path", §The finding worth upstreaming): a 262144-slot pool of one
KV head (head_dim 256) stored as int8 with per-(token,head) scales in side tensors, 16
query heads, 2048 query rows each gathering top-k = 1024 distinct uniform slots. Inputs
are seeded synthetic data (gen.page1_shape, seed 1).

One step = the whole hot path over one batch: quantize-on-write of the step's 2048 new
tokens (qkv_write_int8), then the gather decode attention of the 2048 rows
(qsa_gather_attn; the split-K merge runs too when --splits > 1). The L2 cache is flushed
(a 256 MiB write) between timed steps, outside the timed events.

Metric: gathered-KV GB/s = rows * top-k * (2 * 256 + 2 * 4) bytes per step / step time,
plus rows/s. The same step through the C ABI with host buffers (pinned host -> device
copies of q, indices and new tokens; device -> host copy of the output) gives `e2e`.
`--impl reference` times the CPU oracle on a bounded row sample instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "gathered-KV GB/s (% of GB300 HBM peak) & rows/s, 2048 rows x topk 1024"
ROWS, TOPK, HEAD_DIM, GROUP = 2048, 1024, 256, 16
SLOT_BYTES = {"int8_side": 2 * HEAD_DIM + 8, "int8_inline": 2 * (HEAD_DIM + 4), "e4m3": 2 * HEAD_DIM,
              "bf16": 4 * HEAD_DIM}
L2_FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gather_int8_side_page1_traffic.txt")
KERNEL_SOURCES = ["gather_attn.cuh", "qkv_internal.cuh", "gather_int8_side.cu"]


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    # 2000 steps keep the timed region ~0.6 s long, so the 50 ms clock sampler sees it under load
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--splits", type=int, default=1, help="K-splits of each row (1 = unsplit)")
    ap.add_argument("--no-formats", action="store_true", help="skip the per-format side measurements")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the side measurements of the split-K, long-context and chunked-prefill workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-rows", type=int, default=0, help="oracle rows per sample (0 = auto)")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def _free_port() -> int:
    import socket
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch_ranks(n: int, argv) -> int:
    """Run this script as n ranks on this node (one process per GPU, torch.distributed.run on
    127.0.0.1) and return their exit status. Used when --gpus N > 1 is given without an outer
    launcher; under one, WORLD_SIZE is set and the ranks run directly."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", os.path.abspath(__file__), *argv]
    return subprocess.run(cmd).returncode


def check_world(args) -> bool:
    """True when this process is one rank of the launch --gpus asks for; False when it must
    launch the ranks itself. A launcher whose WORLD_SIZE disagrees with --gpus is refused."""
    if "WORLD_SIZE" in os.environ:
        world = int(os.environ["WORLD_SIZE"])
        if world != args.gpus:
            raise SystemExit(f"bench.py: --gpus {args.gpus} but the launcher started {world} ranks")
        return True
    return args.gpus <= 1


def load_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    """sha256[:16] of the gather kernel's code: its sources with comments and blank lines
    removed, so that an edit of the comments alone keeps the recorded profile valid."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "quantized_kv_cache_write_gb300", "csrc", name)) as f:
            for line in f:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def load_profile():
    """The committed ncu figures of the gather kernel, if taken on the current kernel source."""
    try:
        kv = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256_16") != kernel_source_hash():
            return None
        return kv
    except Exception:
        return None


def load_traffic():
    """ncu dram bytes per gather launch, if taken on the current kernel source; else None."""
    kv = load_profile()
    try:
        return float(kv["dram_bytes_per_launch"]) if kv else None
    except (KeyError, ValueError):
        return None


def max_over_ranks(values, device="cpu"):
    """Elementwise max of per-rank floats (a barrier-synchronised all-reduce; identity at N=1)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(units_per_rank: float, world: int, ms_max: float) -> float:
    """Weak scaling: every rank processes `units_per_rank`; the job takes the slowest rank's time."""
    return world * units_per_rank / (ms_max * 1e-3)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,utilization.gpu")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return self.summarize(out)

    @staticmethod
    def summarize(out: str) -> dict:
        """Median SM clock under load, the max clock and the throttle reasons seen, from the
        sampler's CSV lines (FIELDS order, no header, no units)."""
        rows = []
        for line in out.strip().splitlines():
            p = [x.strip() for x in line.split(",")]
            if len(p) < 7:
                continue
            try:
                rows.append((float(p[0]), float(p[1]), p[2], p[3], p[4], p[5], float(p[6])))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        loaded = [r for r in rows if r[6] > 0] or rows
        sm = sorted(r[0] for r in loaded)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i in range(4) if r[2 + i].lower() == "active"})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": loaded[0][1], "reasons": reasons,
                "samples": len(rows), "samples_under_load": len([r for r in rows if r[6] > 0])}


# ------------------------------------------------------------------ the oracle arm

def oracle_setup(wl):
    from oracle import attention as oatt
    from oracle import quant as oq
    kc, vc, ks, vs = oq.write_int8(wl.k_tokens, wl.v_tokens, wl.slot_mapping, wl.num_slots, "side")
    return oatt.int8_side_pool_fp64(kc, ks), oatt.int8_side_pool_fp64(vc, vs)


_ORACLE = None  # (wl, K, V) shared with forked oracle workers (copy-on-write)


def _oracle_chunk(rows):
    wl, K, V = _ORACLE
    from oracle import attention as oatt
    from oracle import quant as oq
    lo, hi = rows[0], rows[-1] + 1
    oq.int8_quantize(oq.bf16_bits_to_f32(wl.step_k[lo:hi]))
    oq.int8_quantize(oq.bf16_bits_to_f32(wl.step_v[lo:hi]))
    oatt.gather_attention(wl.q, K, V, wl.topk, wl.softmax_scale, rows=rows)
    return len(rows)


def start_oracle_pool(wl):
    """A pool of one forked oracle worker per host core, holding the page-1 workload and its
    fp64 pool (shared copy-on-write). Must be called before the process first uses CUDA."""
    global _ORACLE
    import multiprocessing as mp
    K, V = oracle_setup(wl)
    _ORACLE = (wl, K, V)
    cores = max(1, min(len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count(), 64))
    return mp.get_context("fork").Pool(cores)


def time_oracle_pool(pool, sample_rows: int = 0, repeats: int = 3) -> dict:
    """cpu_baseline: the oracle on every host core over a bounded sample of the page-1 rows
    (32 rows per core: about a second of CPU work per step), mean of `repeats` steps."""
    cores = pool._processes
    n = min(ROWS, sample_rows or 32 * cores)
    per = -(-n // cores)
    chunks = [list(range(i, min(n, i + per))) for i in range(0, n, per)]
    pool.map(_oracle_chunk, chunks)  # warm the workers
    times = []
    for _ in range(repeats):
        t0 = time.perf_counter()
        pool.map(_oracle_chunk, chunks)
        times.append(time.perf_counter() - t0)
    pool.close()
    pool.join()
    sec = sum(times) / len(times)
    return {"value": round(n * TOPK * SLOT_BYTES["int8_side"] / sec / 1e9, 4), "unit": "GB/s", "cores": len(chunks),
            "kind": "oracle", "cpu": cpu_model(),
            "sample": f"first {n} of 2048 rows (and their {n} new tokens) per step, mean of {repeats} steps, fp64 "
                      f"numpy oracle, rows split over {len(chunks)} forked workers with 1 BLAS thread each; "
                      f"{round(n / sec, 1)} rows/s"}


def cpu_model() -> str:
    """The host CPU's model name (lscpu), else the machine type."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


def run_reference(args):
    """The oracle on the host's cores: rows of a bounded sample split over one forked worker
    per core (one BLAS thread each). No GPU is touched in this process, so forking is safe."""
    global _ORACLE
    rank, world, _ = dist_env()
    if rank != 0:
        return
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    os.environ["OMP_NUM_THREADS"] = "1"
    import multiprocessing as mp
    from gen import page1_shape
    wl = page1_shape(1)
    K, V = oracle_setup(wl)
    _ORACLE = (wl, K, V)
    cores = max(1, min(len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count(), 64))
    # rows per step: the whole --steps K --warmup W run stays near a minute of wall time
    # (the oracle takes ~2 ms per row of 1024 keys x 16 heads on one core)
    steps_all = max(1, args.steps) + max(1, args.warmup)
    n = args.cpu_sample_rows or max(cores, min(ROWS, int(60.0 * cores / steps_all / 0.002)))
    per = -(-n // cores)
    chunks = [list(range(i, min(n, i + per))) for i in range(0, n, per)]
    with mp.get_context("fork").Pool(len(chunks)) as pool:
        pool.map(_oracle_chunk, chunks)  # warm the workers
        for _ in range(max(1, args.warmup)):
            pool.map(_oracle_chunk, chunks)
        times = []
        for _ in range(max(1, args.steps)):
            t0 = time.perf_counter()
            pool.map(_oracle_chunk, chunks)
            times.append(time.perf_counter() - t0)
    sec = sum(times) / len(times)
    gbs = n * TOPK * SLOT_BYTES["int8_side"] / sec / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"page-1 shape, oracle sample of {n} of 2048 rows", "rows": ROWS, "topk": TOPK,
                   "num_slots": wl.num_slots, "num_q_heads": GROUP, "num_kv_heads": 1, "head_dim": HEAD_DIM,
                   "format": "int8_side", "parallelism": f"rows over {len(chunks)} CPU worker processes"},
        "rows_per_s": round(n / sec, 2),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": len(chunks), "kind": "oracle",
                         "cpu": cpu_model(),
                         "sample": f"first {n} of 2048 rows (and their {n} new tokens) per step, fp64 numpy oracle, "
                                   f"rows split over {len(chunks)} forked workers with 1 BLAS thread each"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ the GPU arm

def main():
    args = parse_args()
    if args.gpus < 1:
        raise SystemExit("bench.py: --gpus must be >= 1")
    if not check_world(args):
        if args.impl == "ours":
            import torch
            if torch.cuda.device_count() < args.gpus:
                raise SystemExit(f"bench.py: --gpus {args.gpus} but {torch.cuda.device_count()} GPU(s) are visible")
        raise SystemExit(launch_ranks(args.gpus, sys.argv[1:]))
    if args.impl == "reference":
        run_reference(args)
        return
    rank, world, local = dist_env()
    if world > 1 or rank == 0:
        os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
        os.environ.setdefault("OMP_NUM_THREADS", "1")
    import numpy as np
    import torch
    import torch.distributed as dist

    import __graft_entry__
    __graft_entry__.build()
    import quantized_kv_cache_write_gb300 as q
    from gen import page1_shape

    # the CPU baseline's worker pool is forked now, before this process touches the GPU (a
    # process forked after CUDA starts cannot use it, and forking then is unsafe)
    wl = page1_shape(1)
    oracle_pool = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        oracle_pool = start_oracle_pool(wl)

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev_index = torch.cuda.current_device()
    stream = torch.cuda.current_stream()

    # ---- setup (untimed): every rank runs its own page-1 shape problem (weak scaling)
    S, H, D = wl.num_slots, 1, HEAD_DIM
    bf = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    k_tok, v_tok = bf(wl.k_tokens), bf(wl.v_tokens)
    slots_all = torch.from_numpy(wl.slot_mapping).cuda()
    q_dev = bf(wl.q)
    idx = torch.from_numpy(wl.topk).cuda()
    step_k, step_v = bf(wl.step_k), bf(wl.step_v)
    step_slots = torch.from_numpy(wl.step_slots).cuda()
    kc = torch.zeros((S, H, D), dtype=torch.int8, device="cuda")
    vc = torch.zeros_like(kc)
    ks = torch.zeros((S, H), dtype=torch.float32, device="cuda")
    vs = torch.zeros_like(ks)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q.qkv_write_int8(k_tok, v_tok, slots_all, kc, vc, ks, vs, dev_status=status)
    P = args.splits
    out = torch.empty((ROWS, GROUP, D), dtype=torch.float32, device="cuda")
    o_part = torch.empty((ROWS, P, GROUP, D), dtype=torch.float32, device="cuda") if P > 1 else None
    lse_part = torch.empty((ROWS, P, GROUP), dtype=torch.float32, device="cuda") if P > 1 else None
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    def gather(qt, it, ot):
        if P == 1:
            q.qsa_gather_attn(qt, q.QKV_INT8_SIDE, kc, vc, it, wl.softmax_scale, k_scale_tok=ks, v_scale_tok=vs,
                              out=ot, dev_status=status)
        else:
            q.qsa_gather_attn(qt, q.QKV_INT8_SIDE, kc, vc, it, wl.softmax_scale, k_scale_tok=ks, v_scale_tok=vs,
                              num_splits=P, o_part=o_part, lse_part=lse_part, dev_status=status)
            q.qsa_splitk_merge(o_part, lse_part, ot)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        q.qkv_write_int8(step_k, step_v, step_slots, kc, vc, ks, vs, dev_status=status)
        if ev:
            ev[1].record(stream)
        gather(q_dev, idx, out)
        if ev:
            ev[2].record(stream)

    launches_per_step = 2 + (1 if P > 1 else 0)
    for i in range(args.warmup):
        flush.fill_(float(i))
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(dev_index)
    sampler.start()
    time.sleep(0.3)  # let the sampler come up before the timed region
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(float(i))
        step(evs[i])
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    clocks = sampler.stop()
    if world > 1:
        dist.barrier()
    step_ms = [e[0].elapsed_time(e[2]) for e in evs]
    gather_ms = [e[1].elapsed_time(e[2]) for e in evs]
    write_ms = [e[0].elapsed_time(e[1]) for e in evs]
    ms, g_ms = max_over_ranks([sum(step_ms) / len(step_ms), sum(gather_ms) / len(gather_ms)], device="cuda")
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item()} during the benchmark")

    gathered = ROWS * TOPK * SLOT_BYTES["int8_side"]
    value = whole_job_rate(gathered, world, ms) / 1e9
    rows_per_s = whole_job_rate(ROWS, world, ms)
    peak, peak_src = load_peak()
    achieved = gathered / (g_ms * 1e-3) / 1e9
    uniq_slots = int(np.unique(wl.topk).size)
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8 codes -> fp16 mma, fp32 accumulate", "data": "synthetic",
        "config": {"workload": "page-1 shape: 2048 rows x top-k 1024 over a 262144-slot int8 pool "
                               "(side-tensor scales), 1 KV head, 16 query heads, head_dim 256, seed 1",
                   "rows": ROWS, "topk": TOPK, "num_slots": S, "num_q_heads": GROUP, "num_kv_heads": 1,
                   "head_dim": HEAD_DIM, "format": "int8_side", "num_splits": P,
                   "step": "qkv_write_int8 of 2048 new tokens + qsa_gather_attn" + (" + qsa_splitk_merge" if P > 1 else ""),
                   "l2": "flushed (256 MiB write) between timed steps", "parallelism": f"dp{world} (independent problems)"},
        "rows_per_s": round(rows_per_s, 1),
        "frac_of_hbm_peak_total": round(value / (world * peak), 4),
        "unique_gathered_GBps": round(world * uniq_slots * SLOT_BYTES["int8_side"] / (ms * 1e-3) / 1e9, 2),
        "frac_of_hbm_peak_unique": round(uniq_slots * SLOT_BYTES["int8_side"] / (ms * 1e-3) / 1e9 / peak, 4),
        "unique_slots": uniq_slots,
        "write_ms": round(sum(write_ms) / len(write_ms), 5),
        "gather_ms": round(g_ms, 5),
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": load_traffic(),
                     "kernel": "gather_attn_kernel<QKV_INT8_SIDE>",
                     "algorithmic_bytes_per_launch": gathered, "peak_source": peak_src,
                     "ncu": ({k: float(v) for k, v in prof.items() if k not in ("kernel_source_sha256_16",)}
                             if (prof := load_profile()) else None)},
        "wall_s_timed_region": round(t_wall, 3),
        "pages_context": {"gb10_side_ms": 9.6, "gb10_inline_ms": 60.2,
                          "note": "one GB10 (sm_121), Triton path; context only"},
    }

    # ---- end to end through the public API with host buffers
    pin = lambda t: t.cpu().pin_memory()
    h_q, h_idx, h_k, h_v, h_slots = pin(q_dev), pin(idx), pin(step_k), pin(step_v), pin(step_slots)
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    d_q, d_idx = torch.empty_like(q_dev), torch.empty_like(idx)
    d_k, d_v, d_slots = torch.empty_like(step_k), torch.empty_like(step_v), torch.empty_like(step_slots)
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_idx, h_k, h_v, h_slots))
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step():
        d_q.copy_(h_q, non_blocking=True)
        d_idx.copy_(h_idx, non_blocking=True)
        d_k.copy_(h_k, non_blocking=True)
        d_v.copy_(h_v, non_blocking=True)
        d_slots.copy_(h_slots, non_blocking=True)
        q.qkv_write_int8(d_k, d_v, d_slots, kc, vc, ks, vs, dev_status=status)
        gather(d_q, d_idx, out)
        h_out.copy_(out, non_blocking=True)

    n_e2e = max(3, min(args.steps, 50))
    for i in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_ms = []
    for i in range(n_e2e):
        flush.fill_(float(i))
        e0.record(stream)
        e2e_step()
        e1.record(stream)
        e1.synchronize()
        e_ms.append(e0.elapsed_time(e1))
    em_seq = max_over_ranks([sum(e_ms) / len(e_ms)], device="cuda")[0]

    # The same steps pipelined the way a serving loop runs them: step i's inputs go up on a
    # copy stream while step i - 1 computes, and step i - 1's output comes down on a third
    # stream; inputs and outputs are double-buffered. Every step still copies its own inputs
    # from pinned host memory and reads its output back inside the timed region. No L2 flush:
    # a step's working set (136 MB of distinct pool slots gathered, plus q, indices, output and
    # new tokens) exceeds the 129 MB L2 by itself.
    n_pipe = max(10, min(args.steps, 200))
    ms_pipe = max_over_ranks([e2e_pipelined(q, gather, kc, vc, ks, vs, status, (h_q, h_idx, h_k, h_v, h_slots),
                                            h_out, n_pipe)], device="cuda")[0]
    result["e2e"] = {"value": round(whole_job_rate(gathered, world, ms_pipe) / 1e9, 2), "unit": "GB/s",
                     "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_pipe, 4),
                     "steps": n_pipe, "mode": "pipelined: copies on their own streams, double-buffered",
                     "l2": "not flushed: per-step working set above the L2 size",
                     "sequential": {"value": round(whole_job_rate(gathered, world, em_seq) / 1e9, 2),
                                    "ms_per_step": round(em_seq, 4), "steps": n_e2e,
                                    "l2": "flushed (256 MiB write) before each step, outside the events"}}

    # ---- the other formats, same shape (gather alone; context for the side-vs-inline and
    #      int8-vs-fp8-vs-bf16 comparisons of the pages)
    if not args.no_formats and rank == 0:
        result["formats"] = measure_formats(q, wl, q_dev, idx, flush, stream, max(5, min(args.steps, 30)), peak)

    if not args.no_workloads and rank == 0:
        result["workloads"] = measure_workloads(q, flush, stream, max(5, min(args.steps, 20)), peak)

    if oracle_pool is not None:
        result["cpu_baseline"] = time_oracle_pool(oracle_pool, args.cpu_sample_rows)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


def e2e_pipelined(q, gather, kc, vc, ks, vs, status, host_inputs, h_out_proto, n):
    """Mean ms per step of n decode steps through the public API with host buffers, pipelined.

    Step i: h2d of its q, indices and new tokens on a copy stream; on the compute stream the
    write of the new tokens and the gather, once that copy is in and the output buffer's
    previous d2h is out; then the d2h of its output on a third stream. Two buffer sets.
    """
    import torch
    h_q, h_idx, h_k, h_v, h_slots = host_inputs
    cs, hs, ds = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    bufs = [dict(q=torch.empty(h_q.shape, dtype=h_q.dtype, device="cuda"),
                 idx=torch.empty(h_idx.shape, dtype=h_idx.dtype, device="cuda"),
                 k=torch.empty(h_k.shape, dtype=h_k.dtype, device="cuda"),
                 v=torch.empty(h_v.shape, dtype=h_v.dtype, device="cuda"),
                 slots=torch.empty(h_slots.shape, dtype=h_slots.dtype, device="cuda"),
                 out=torch.empty(h_out_proto.shape, dtype=h_out_proto.dtype, device="cuda")) for _ in range(2)]
    h_outs = [torch.empty(h_out_proto.shape, dtype=h_out_proto.dtype).pin_memory() for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def run(steps):
        for i in range(steps):
            b = bufs[i % 2]
            with torch.cuda.stream(hs):
                if i >= 2:
                    hs.wait_event(ev_comp[i % 2])  # step i - 2 has read these inputs
                b["q"].copy_(h_q, non_blocking=True)
                b["idx"].copy_(h_idx, non_blocking=True)
                b["k"].copy_(h_k, non_blocking=True)
                b["v"].copy_(h_v, non_blocking=True)
                b["slots"].copy_(h_slots, non_blocking=True)
                ev_in[i % 2].record(hs)
            with torch.cuda.stream(cs):
                cs.wait_event(ev_in[i % 2])
                if i >= 2:
                    cs.wait_event(ev_out[i % 2])  # step i - 2's output has been read back
                q.qkv_write_int8(b["k"], b["v"], b["slots"], kc, vc, ks, vs, dev_status=status)
                gather(b["q"], b["idx"], b["out"])
                ev_comp[i % 2].record(cs)
            with torch.cuda.stream(ds):
                ds.wait_event(ev_comp[i % 2])
                h_outs[i % 2].copy_(b["out"], non_blocking=True)
                ev_out[i % 2].record(ds)

    run(4)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(cs)
    hs.wait_event(start)
    ds.wait_event(start)
    run(n)
    cs.wait_stream(hs)
    cs.wait_stream(ds)
    end.record(cs)
    end.synchronize()
    return start.elapsed_time(end) / n


def measure_formats(q, wl, q_dev, idx, flush, stream, steps, peak):
    import numpy as np
    import torch
    S, D = wl.num_slots, HEAD_DIM
    bf = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    k_tok, v_tok = bf(wl.k_tokens), bf(wl.v_tokens)
    slots = torch.from_numpy(wl.slot_mapping).cuda()
    out = torch.empty((ROWS, GROUP, D), dtype=torch.float32, device="cuda")
    res = {}
    for fmt in ("int8_side", "int8_inline", "e4m3", "bf16"):
        kw = {}
        if fmt == "int8_side":
            kc = torch.zeros((S, 1, D), dtype=torch.int8, device="cuda")
            vc = torch.zeros_like(kc)
            ks = torch.zeros((S, 1), dtype=torch.float32, device="cuda")
            vs = torch.zeros_like(ks)
            q.qkv_write_int8(k_tok, v_tok, slots, kc, vc, ks, vs)
            kw = dict(k_scale_tok=ks, v_scale_tok=vs)
        elif fmt == "int8_inline":
            kc = torch.zeros((S, 1, D + 4), dtype=torch.uint8, device="cuda")
            vc = torch.zeros_like(kc)
            q.qkv_write_int8(k_tok, v_tok, slots, kc, vc, layout=q.QKV_INT8_INLINE)
        elif fmt == "e4m3":
            amax = torch.zeros(1, dtype=torch.int32, device="cuda")
            sc = torch.zeros(2, dtype=torch.float32, device="cuda")
            q.qkv_e4m3_calibrate(k_tok, amax, sc[0:1])
            q.qkv_e4m3_calibrate(v_tok, amax, sc[1:2])
            ksl, vsl = sc.tolist()
            kc = torch.zeros((S, 1, D), dtype=torch.uint8, device="cuda")
            vc = torch.zeros_like(kc)
            q.qkv_write_e4m3(k_tok, v_tok, slots, kc, vc, ksl, vsl)
            kw = dict(k_scale_layer=ksl, v_scale_layer=vsl)
        else:
            kc = torch.zeros((S, 1, D), dtype=torch.bfloat16, device="cuda")
            vc = torch.zeros_like(kc)
            kc[slots] = k_tok
            vc[slots] = v_tok
        code = q.FORMATS[fmt]
        for i in range(3):
            q.qsa_gather_attn(q_dev, code, kc, vc, idx, wl.softmax_scale, out=out, **kw)
        ms = []
        for i in range(steps):
            flush.fill_(float(i))
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            q.qsa_gather_attn(q_dev, code, kc, vc, idx, wl.softmax_scale, out=out, **kw)
            b.record(stream)
            b.synchronize()
            ms.append(a.elapsed_time(b))
        m = sum(ms) / len(ms)
        gbs = ROWS * TOPK * SLOT_BYTES[fmt] / (m * 1e-3) / 1e9
        res[fmt] = {"gather_ms": round(m, 5), "gathered_GBps": round(gbs, 2), "frac_of_hbm_peak": round(gbs / peak, 4),
                    "rows_per_s": round(ROWS / (m * 1e-3), 1), "bytes_per_slot": SLOT_BYTES[fmt]}
        # the other engines of the same gather: the resident-grid scheduler (every format) and
        # q.K^T on tcgen05 with tensor-memory operands (int8 side only)
        sched = torch.zeros(2, dtype=torch.int32, device="cuda")
        engines = {"persistent": q.QSA_ENGINE_PERSISTENT}
        if fmt == "int8_side":
            engines["tcgen05"] = q.QSA_ENGINE_TCGEN05
        for name, eng in engines.items():
            t = _time_events(lambda eng=eng: q.qsa_gather_attn_ex(
                q_dev, code, kc, vc, idx, wl.softmax_scale, out=out, engine=eng,
                sched=sched if eng == q.QSA_ENGINE_PERSISTENT else None, **kw), flush, stream, steps)
            g2 = ROWS * TOPK * SLOT_BYTES[fmt] / (t * 1e-3) / 1e9
            res[fmt][name + "_engine"] = {"gather_ms": round(t, 5), "gathered_GBps": round(g2, 2),
                                          "frac_of_hbm_peak": round(g2 / peak, 4)}
        del kc, vc
        torch.cuda.empty_cache()
    return res


def _device_pool(q, wl, fmt):
    """Write a workload's tokens into a device pool with the library's own write kernels."""
    import numpy as np
    import torch
    S, H, D = wl.num_slots, wl.num_kv_heads, HEAD_DIM
    bf = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    k_tok, v_tok = bf(wl.k_tokens), bf(wl.v_tokens)
    slots = torch.from_numpy(wl.slot_mapping).cuda()
    if fmt == "int8_side":
        kc = torch.zeros((S, H, D), dtype=torch.int8, device="cuda")
        vc = torch.zeros_like(kc)
        ks = torch.zeros((S, H), dtype=torch.float32, device="cuda")
        vs = torch.zeros_like(ks)
        q.qkv_write_int8(k_tok, v_tok, slots, kc, vc, ks, vs)
        return kc, vc, dict(k_scale_tok=ks, v_scale_tok=vs), 1.0
    amax = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc = torch.zeros(2, dtype=torch.float32, device="cuda")
    q.qkv_e4m3_calibrate(k_tok, amax, sc[0:1])
    q.qkv_e4m3_calibrate(v_tok, amax, sc[1:2])
    ksl, vsl = sc.tolist()
    kc = torch.zeros((S, H, D), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    q.qkv_write_e4m3(k_tok, v_tok, slots, kc, vc, ksl, vsl)
    return kc, vc, dict(k_scale_layer=ksl, v_scale_layer=vsl), vsl


def _time_events(fn, flush, stream, reps):
    """Mean device time of fn() in ms (CUDA events on `stream`), L2 flushed before every rep."""
    import torch
    for _ in range(3):
        fn()
    ms = []
    for i in range(reps):
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    return sum(ms) / len(ms)


def _time_graph(fn, flush, stream, reps):
    """Mean device time in ms of one replay of a CUDA graph captured from fn() (L2 flushed
    before every replay). fn runs eagerly first, on the capture's side stream too."""
    import torch
    fn()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    ms = _time_events(g.replay, flush, stream, reps)
    del g
    return ms


def measure_l2_roof(stream, reps=20):
    """An L2 bandwidth roof: the best of torch's sum (a read) and copy (a read plus a write) over
    buffers of 16 to 64 MiB, well inside the 129 MB L2, each warmed once and then timed with
    CUDA events (no flush: the point is to stay in L2). GB/s of bytes moved."""
    import torch
    best = {"sum": 0.0, "copy": 0.0}
    for mib in (16, 32, 64):
        n = (mib << 20) // 4
        a = torch.ones(n, dtype=torch.float32, device="cuda")
        b = torch.empty_like(a)
        for name, fn, nbytes in (("sum", lambda: a.sum(), 4 * n), ("copy", lambda: b.copy_(a), 8 * n)):
            fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
            e1.synchronize()
            best[name] = max(best[name], nbytes * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9)
        del a, b
    torch.cuda.empty_cache()
    return {"GBps": round(max(best.values()), 1), "read_GBps": round(best["sum"], 1),
            "copy_GBps": round(best["copy"], 1),
            "how": "best of torch sum (read) and copy (read + write) over 16-64 MiB L2-resident buffers"}


def measure_workloads(q, flush, stream, reps, peak):
    """The pages' other workload shapes, gather path only (context; the metric is the page-1 shape).

    split-K workloads: the split gather followed by qsa_splitk_merge (two launches) against
    qsa_gather_attn_splitk_fused (one launch); chunked prefill: the 8192-token writes and the
    8192-row causal gather, whose 4.3 MB of distinct slots stay in L2.
    """
    import numpy as np
    import torch
    from gen import E4M3_SPLITK_LAYERS, chunked_prefill, e4m3_splitk_layer, long_context_decode
    res = {}

    def split_variants(wl, fmt, kc, vc, kw, vpost):
        R, Hq, D, P = wl.rows, wl.num_q_heads, HEAD_DIM, wl.num_splits
        qd = torch.from_numpy(np.ascontiguousarray(wl.q).view(np.int16)).view(torch.bfloat16).cuda()
        idx = torch.from_numpy(np.ascontiguousarray(wl.topk, dtype=np.int32)).cuda()
        out = torch.empty((R, Hq, D), dtype=torch.float32, device="cuda")
        o_part = torch.empty((R, P, Hq, D), dtype=torch.float32, device="cuda")
        lse_part = torch.empty((R, P, Hq), dtype=torch.float32, device="cuda")
        counters = torch.zeros((R, wl.num_kv_heads), dtype=torch.int32, device="cuda")
        code = q.FORMATS[fmt]

        def two():
            q.qsa_gather_attn(qd, code, kc, vc, idx, wl.softmax_scale, num_splits=P, o_part=o_part,
                              lse_part=lse_part, **kw)
            q.qsa_splitk_merge(o_part, lse_part, out, v_scale_post=vpost)

        def fused():
            q.qsa_gather_attn_splitk_fused(qd, code, kc, vc, idx, wl.softmax_scale, num_splits=P, out=out,
                                           o_part=o_part, lse_part=lse_part, counters=counters, **kw)

        def unsplit():
            q.qsa_gather_attn(qd, code, kc, vc, idx, wl.softmax_scale, out=out, **kw)

        # the split count qsa_suggest_num_splits picks (one wave of resident CTAs), fused
        Pa = q.qsa_suggest_num_splits(code, R, Hq, wl.num_kv_heads, wl.topk.shape[1])
        o_pa = torch.empty((R, Pa, Hq, D), dtype=torch.float32, device="cuda")
        l_pa = torch.empty((R, Pa, Hq), dtype=torch.float32, device="cuda")
        cnt_a = torch.zeros((R, wl.num_kv_heads), dtype=torch.int32, device="cuda")

        def fused_suggested():
            q.qsa_gather_attn_splitk_fused(qd, code, kc, vc, idx, wl.softmax_scale, num_splits=Pa, out=out,
                                           o_part=o_pa, lse_part=l_pa, counters=cnt_a, **kw)

        t = {"split_plus_merge_ms": _time_events(two, flush, stream, reps),
             "fused_ms": _time_events(fused, flush, stream, reps),
             "unsplit_ms": _time_events(unsplit, flush, stream, reps)}
        return t, (qd, idx, out), {"fused": fused, "fused_suggested": fused_suggested, "suggested_splits": Pa}

    # calibrated E4M3 split-K: 12 layers, each its own 131072-slot pool
    per_layer, fns = [], []
    for layer in range(E4M3_SPLITK_LAYERS):
        wl = e4m3_splitk_layer(layer)
        kc, vc, kw, vpost = _device_pool(q, wl, "e4m3")
        t, _, f = split_variants(wl, "e4m3", kc, vc, kw, vpost)
        per_layer.append(t)
        fns.append(f)  # keeps this layer's pool and buffers alive for the graph below
        del kc, vc
    tot = {k: sum(t[k] for t in per_layer) for k in per_layer[0]}
    bytes_layer = 64 * 2051 * SLOT_BYTES["e4m3"]
    # all 12 layers' fused launches as one CUDA graph, replayed after one L2 flush: a decode
    # step's attention over the layers without a host launch or an event between layers
    graph = {}
    for name in ("fused", "fused_suggested"):
        graph[name + "_ms"] = _time_graph(lambda name=name: [f[name]() for f in fns], flush, stream, reps)
    res["e4m3_splitk_12_layers"] = {
        "shape": "12 layers x (64 rows, top-k 2051, 8 splits) over 131072-slot E4M3 pools, 16 query heads",
        "sum_ms": {k: round(v, 5) for k, v in tot.items()},
        "per_layer_ms": {k: [round(t[k], 5) for t in per_layer] for k in per_layer[0]},
        "fused_gathered_GBps": round(E4M3_SPLITK_LAYERS * bytes_layer / (tot["fused_ms"] * 1e-3) / 1e9, 2),
        "note": "each layer timed alone after an L2 flush",
        "graph_12_layers_ms": {k: round(v, 5) for k, v in graph.items()},
        "graph_suggested_splits": fns[0]["suggested_splits"],
        "graph_fused_gathered_GBps": round(E4M3_SPLITK_LAYERS * bytes_layer / (graph["fused_ms"] * 1e-3) / 1e9, 2),
        "graph_fused_suggested_gathered_GBps": round(
            E4M3_SPLITK_LAYERS * bytes_layer / (graph["fused_suggested_ms"] * 1e-3) / 1e9, 2),
        "graph_note": "one CUDA graph of the 12 layers' fused launches, L2 flushed once before each replay"}
    del fns

    # mixed decode batches: rows of very different lengths in one varlen launch with the fused
    # split-K merge, on the default grid (one CTA per work item) and on the persistent grid
    from gen import bulk_tail_decode, mixed_catchup_decode
    mixed = {}
    for wname, make in (("catchup_46_plus_decode_3", mixed_catchup_decode), ("bulk_48_plus_tail_13", bulk_tail_decode)):
        wl = make()
        lens = torch.from_numpy(wl.row_len).cuda()
        visits = int(wl.row_len.sum())
        entry = {"shape": wl.name, "key_visits": visits}
        for fmt in ("e4m3", "int8_side"):
            kc, vc, kw, _ = _device_pool(q, wl, fmt)
            qd = torch.from_numpy(np.ascontiguousarray(wl.q).view(np.int16)).view(torch.bfloat16).cuda()
            idx = torch.from_numpy(np.ascontiguousarray(wl.topk, dtype=np.int32)).cuda()
            R, Hq, D = wl.rows, wl.num_q_heads, HEAD_DIM
            code = q.FORMATS[fmt]
            Pa = q.qsa_suggest_num_splits(code, R, Hq, wl.num_kv_heads, wl.topk.shape[1])
            sched = torch.zeros(2, dtype=torch.int32, device="cuda")
            t = {"suggested_splits": Pa}
            for P in sorted({8, Pa}):
                out = torch.empty((R, Hq, D), dtype=torch.float32, device="cuda")
                o_part = torch.empty((R, P, Hq, D), dtype=torch.float32, device="cuda")
                lse_part = torch.empty((R, P, Hq), dtype=torch.float32, device="cuda")
                cnt = torch.zeros((R, 1, 1), dtype=torch.int32, device="cuda")
                for ename, eng in (("default", q.QSA_ENGINE_DEFAULT), ("persistent", q.QSA_ENGINE_PERSISTENT)):
                    t[f"fused_P{P}_{ename}_ms"] = round(_time_events(lambda eng=eng, P=P, out=out, o_part=o_part,
                                                                      lse_part=lse_part, cnt=cnt: q.qsa_gather_attn_ex(
                        qd, code, kc, vc, idx, wl.softmax_scale, num_splits=P, out=out, o_part=o_part,
                        lse_part=lse_part, counters=cnt, topk_len=lens, engine=eng,
                        sched=sched if eng == q.QSA_ENGINE_PERSISTENT else None, **kw), flush, stream, reps), 5)
            entry[fmt] = t
            del kc, vc
        mixed[wname] = entry
    mixed["note"] = ("varlen + fused split-K merge in one launch; default = one CTA per (row, split) item, "
                     "persistent = resident CTAs taking items from an atomic counter; L2 flushed before each launch")
    res["mixed_decode"] = mixed
    torch.cuda.empty_cache()

    # long-context decode: 8 x 131072 tokens, 40 rows x top-k 2048, 16 splits; also the paged kernel
    wl = long_context_decode(3)
    kc, vc, kw, vpost = _device_pool(q, wl, "int8_side")
    t, (qd, idx, out), _ = split_variants(wl, "int8_side", kc, vc, kw, vpost)
    table = torch.from_numpy(np.ascontiguousarray(wl.block_table, dtype=np.int32)).cuda()
    rs = torch.from_numpy(np.ascontiguousarray(wl.row_seq, dtype=np.int32)).cuda()
    pos = torch.from_numpy(np.ascontiguousarray(wl.topk_pos, dtype=np.int32)).cuda()
    P = wl.num_splits
    o_part = torch.empty((wl.rows, P, wl.num_q_heads, HEAD_DIM), dtype=torch.float32, device="cuda")
    lse_part = torch.empty((wl.rows, P, wl.num_q_heads), dtype=torch.float32, device="cuda")

    def paged():
        q.qsa_gather_attn_paged(qd, q.QKV_INT8_SIDE, kc, vc, table, rs, pos, wl.block_size, wl.softmax_scale,
                                num_splits=P, o_part=o_part, lse_part=lse_part, **kw)
        q.qsa_splitk_merge(o_part, lse_part, out)

    t["paged_split_plus_merge_ms"] = _time_events(paged, flush, stream, reps)
    # the split count qsa_suggest_num_splits picks for this shape (one wave of resident CTAs)
    Pa = q.qsa_suggest_num_splits(q.QKV_INT8_SIDE, wl.rows, wl.num_q_heads, wl.num_kv_heads, wl.topk.shape[1])
    o_pa = torch.empty((wl.rows, Pa, wl.num_q_heads, HEAD_DIM), dtype=torch.float32, device="cuda")
    l_pa = torch.empty((wl.rows, Pa, wl.num_q_heads), dtype=torch.float32, device="cuda")
    cnt = torch.zeros((wl.rows, 1, 1), dtype=torch.int32, device="cuda")
    t["fused_suggested_splits_ms"] = _time_events(
        lambda: q.qsa_gather_attn_splitk_fused(qd, q.QKV_INT8_SIDE, kc, vc, idx, wl.softmax_scale, num_splits=Pa,
                                               out=out, o_part=o_pa, lse_part=l_pa, counters=cnt, **kw),
        flush, stream, reps)
    t["suggested_splits"] = Pa
    bytes_lc = wl.rows * wl.topk.shape[1] * SLOT_BYTES["int8_side"]
    res["long_context_decode"] = {
        "shape": "8 seq x 131072 tokens (paged, blocks of 16), 40 rows x top-k 2048, 16 splits, int8 side",
        **{k: (round(v, 5) if isinstance(v, float) else v) for k, v in t.items()},
        "fused_gathered_GBps": round(bytes_lc / (t["fused_ms"] * 1e-3) / 1e9, 2),
        "fused_suggested_gathered_GBps": round(bytes_lc / (t["fused_suggested_splits_ms"] * 1e-3) / 1e9, 2),
        "rows_per_s_suggested": round(wl.rows / (t["fused_suggested_splits_ms"] * 1e-3), 1),
        "note": "42.6 MB gathered per step: launch latency and the wave tail dominate"}
    del kc, vc
    torch.cuda.empty_cache()

    # chunked prefill: 8192 new tokens written, then 8192 causal rows of up to 1024 entries
    wl = chunked_prefill(4)
    bf = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    k_tok, v_tok = bf(wl.k_tokens), bf(wl.v_tokens)
    slots = torch.from_numpy(wl.slot_mapping).cuda()
    S, D = wl.num_slots, HEAD_DIM
    kc = torch.zeros((S, 1, D), dtype=torch.int8, device="cuda")
    vc = torch.zeros_like(kc)
    ks = torch.zeros((S, 1), dtype=torch.float32, device="cuda")
    vs = torch.zeros_like(ks)
    ec = torch.zeros((S, 1, D), dtype=torch.uint8, device="cuda")
    evc = torch.zeros_like(ec)
    w8 = _time_events(lambda: q.qkv_write_int8(k_tok, v_tok, slots, kc, vc, ks, vs), flush, stream, reps)
    we = _time_events(lambda: q.qkv_write_e4m3(k_tok, v_tok, slots, ec, evc, 0.01, 0.01), flush, stream, reps)
    qd = bf(wl.q)
    idx = torch.from_numpy(np.ascontiguousarray(wl.topk, dtype=np.int32)).cuda()
    out = torch.empty((wl.rows, wl.num_q_heads, D), dtype=torch.float32, device="cuda")
    g = _time_events(lambda: q.qsa_gather_attn(qd, q.QKV_INT8_SIDE, kc, vc, idx, wl.softmax_scale, out=out,
                                               k_scale_tok=ks, v_scale_tok=vs), flush, stream, reps)
    lens = torch.from_numpy(np.minimum(np.arange(wl.rows), wl.topk.shape[1]).astype(np.int32)).cuda()
    gv = _time_events(lambda: q.qsa_gather_attn_varlen(qd, q.QKV_INT8_SIDE, kc, vc, idx, lens, wl.softmax_scale,
                                                       out=out, k_scale_tok=ks, v_scale_tok=vs), flush, stream, reps)
    visits = int((wl.topk >= 0).sum())
    l2 = measure_l2_roof(stream)
    res["chunked_prefill"] = {
        "shape": "8192 new tokens into a 524288-slot pool; 8192 rows, row i attends min(1024, i) earlier tokens",
        "write_int8_ms": round(w8, 5), "write_e4m3_ms": round(we, 5),
        "write_int8_GBps": round(8192 * (1024 + 520) / (w8 * 1e-3) / 1e9, 2),
        "gather_int8_side_ms": round(g, 5), "gather_varlen_ms": round(gv, 5), "slot_visits": visits,
        "gather_GBps": round(visits * SLOT_BYTES["int8_side"] / (g * 1e-3) / 1e9, 2),
        "gather_varlen_GBps": round(visits * SLOT_BYTES["int8_side"] / (gv * 1e-3) / 1e9, 2),
        "l2_roof": l2,
        "gather_varlen_frac_of_l2_roof": round(visits * SLOT_BYTES["int8_side"] / (gv * 1e-3) / 1e9 / l2["GBps"], 4),
        "note": "the 8192 written slots (4.3 MB) stay in L2: gathered GB/s is bounded by L2, not HBM "
                f"(measured HBM peak {peak} GB/s; L2 roof measured here)"}
    del kc, vc, ec, evc
    torch.cuda.empty_cache()

    # calibration statistics of one layer's K tensor (the E4M3 split-K layer 0 pool, 67 MB of
    # bf16): the histogram pass is HBM-bound at 2 B per element; the stats pass reads 256 KB
    wl = e4m3_splitk_layer(0)
    x = bf(wl.k_tokens)
    hist = torch.zeros(q.CALIB_BINS, dtype=torch.int64, device="cuda")
    rec = torch.zeros(8, dtype=torch.int64, device="cuda")
    h_ms = _time_events(lambda: q.qkv_calib_histogram(x, hist), flush, stream, reps)
    s_ms = _time_events(lambda: q.qkv_calib_stats(hist, rec), flush, stream, reps)
    amax = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc = torch.zeros(1, dtype=torch.float32, device="cuda")
    a_ms = _time_events(lambda: q.qkv_e4m3_calibrate(x, amax, sc), flush, stream, reps)
    res["calibration"] = {
        "shape": f"one layer's K: {x.numel()} bf16 values (131072 slots x 256)",
        "histogram_ms": round(h_ms, 5), "stats_ms": round(s_ms, 5),
        "histogram_GBps": round(x.numel() * 2 / (h_ms * 1e-3) / 1e9, 2),
        "histogram_frac_of_hbm_peak": round(x.numel() * 2 / (h_ms * 1e-3) / 1e9 / peak, 4),
        "e4m3_calibrate_ms": round(a_ms, 5),
        "e4m3_calibrate_GBps": round(x.numel() * 2 / (a_ms * 1e-3) / 1e9, 2),
        "e4m3_calibrate_frac_of_hbm_peak": round(x.numel() * 2 / (a_ms * 1e-3) / 1e9 / peak, 4)}
    del x

    # the generalisations at the page-1 shape (2048 rows x top-k 1024 over 262144 int8-side slots):
    # head_dim 128, fp16 activations, and a GQA group of 32 query heads (two 16-head CTAs per row)
    from gen import small_random
    variants = {}
    for name, kw in (("head_dim_128", dict(head_dim=128)), ("fp16_activations", dict(act_dtype="f16")),
                     ("gqa_32", dict(num_q_heads=32))):
        wl = small_random(11, num_slots=262144, rows=2048, topk=1024, outlier_frac=0.01, **kw)
        Dv, Sv, Hv = wl.head_dim, wl.num_slots, wl.num_kv_heads
        dt = torch.float16 if wl.act_dtype == "f16" else torch.bfloat16
        tok = lambda b, dt=dt: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(dt).cuda()
        kcv = torch.zeros((Sv, Hv, Dv), dtype=torch.int8, device="cuda")
        vcv = torch.zeros_like(kcv)
        ksv = torch.zeros((Sv, Hv), dtype=torch.float32, device="cuda")
        vsv = torch.zeros_like(ksv)
        q.qkv_write_int8(tok(wl.k_tokens), tok(wl.v_tokens), torch.from_numpy(wl.slot_mapping).cuda(), kcv, vcv,
                         ksv, vsv)
        qv = tok(wl.q)
        iv = torch.from_numpy(np.ascontiguousarray(wl.topk, dtype=np.int32)).cuda()
        ov = torch.empty((wl.rows, wl.num_q_heads, Dv), dtype=torch.float32, device="cuda")
        t = _time_events(lambda: q.qsa_gather_attn(qv, q.QKV_INT8_SIDE, kcv, vcv, iv, wl.softmax_scale, out=ov,
                                                   k_scale_tok=ksv, v_scale_tok=vsv), flush, stream, reps)
        nb = wl.rows * wl.topk.shape[1] * (2 * Dv + 8)
        variants[name] = {"gather_ms": round(t, 5), "gathered_GBps": round(nb / (t * 1e-3) / 1e9, 2),
                          "frac_of_hbm_peak": round(nb / (t * 1e-3) / 1e9 / peak, 4),
                          "num_q_heads": wl.num_q_heads, "head_dim": Dv, "activations": wl.act_dtype}
        del kcv, vcv, ksv, vsv, qv, iv, ov
    variants["note"] = ("int8 side pools, 2048 rows x top-k 1024 over 262144 slots; GB/s over each row's gathered "
                        "bytes once (the GQA-32 rows gather every slot twice, once per 16-head CTA)")
    res["variants"] = variants
    torch.cuda.empty_cache()

    # pool fill: the page-1 pool's 262144 new tokens written in one call (HBM-bound at this size;
    # per token 1024 B of bf16 K and V read, 2 x 260 B (int8 + scale) or 2 x 256 B (E4M3) written)
    from gen import page1_shape
    wl = page1_shape(1, with_step=False)
    k_tok, v_tok = bf(wl.k_tokens), bf(wl.v_tokens)
    slots = torch.from_numpy(wl.slot_mapping).cuda()
    T, S = wl.k_tokens.shape[0], wl.num_slots
    kc = torch.zeros((S, 1, HEAD_DIM), dtype=torch.int8, device="cuda")
    vc = torch.zeros_like(kc)
    ks = torch.zeros((S, 1), dtype=torch.float32, device="cuda")
    vs = torch.zeros_like(ks)
    w8 = _time_events(lambda: q.qkv_write_int8(k_tok, v_tok, slots, kc, vc, ks, vs), flush, stream, reps)
    # the same tokens through a paged pool: one sequence, position t, blocks of 16 in a random
    # physical order (qkv_write_ex), so each token's slot comes from the block table
    B = 16
    perm = np.random.default_rng(5).permutation(S // B).astype(np.int32)
    table = torch.from_numpy(perm.reshape(1, -1)).cuda()
    tseq = torch.zeros(T, dtype=torch.int32, device="cuda")
    tpos = torch.arange(T, dtype=torch.int32, device="cuda")
    w8p = _time_events(lambda: q.qkv_write_ex(k_tok, v_tok, q.QKV_INT8_SIDE, kc, vc, token_seq=tseq, token_pos=tpos,
                                              block_table=table, block_size=B, k_scale=ks, v_scale=vs),
                       flush, stream, reps)
    del kc, vc, ks, vs
    ec = torch.zeros((S, 1, HEAD_DIM), dtype=torch.uint8, device="cuda")
    evc = torch.zeros_like(ec)
    we = _time_events(lambda: q.qkv_write_e4m3(k_tok, v_tok, slots, ec, evc, 0.01, 0.01), flush, stream, reps)
    b8, be = T * (1024 + 520), T * (1024 + 512)
    res["pool_fill"] = {
        "shape": f"{T} bf16 tokens (1 KV head x 256, K and V) written into a {S}-slot pool in one call",
        "write_int8_side_ms": round(w8, 5), "write_e4m3_ms": round(we, 5),
        "write_int8_side_paged_ms": round(w8p, 5),
        "write_int8_side_paged_GBps": round(b8 / (w8p * 1e-3) / 1e9, 2),
        "write_int8_side_GBps": round(b8 / (w8 * 1e-3) / 1e9, 2),
        "write_e4m3_GBps": round(be / (we * 1e-3) / 1e9, 2),
        "write_int8_side_frac_of_hbm_peak": round(b8 / (w8 * 1e-3) / 1e9 / peak, 4),
        "write_e4m3_frac_of_hbm_peak": round(be / (we * 1e-3) / 1e9 / peak, 4)}
    del ec, evc, k_tok, v_tok
    torch.cuda.empty_cache()
    return res


if __name__ == "__main__":
    main()

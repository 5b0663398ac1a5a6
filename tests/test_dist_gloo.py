"""The benchmark's multi-rank host logic on CPU: two gloo ranks (no GPU, no NCCL).

Rows shard across GPUs with no collective on the data path (weak scaling); the only
collectives are the benchmark's barrier and the max of per-rank step times, from which the
whole-job rate is computed.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env()[:2] == (rank, world)
        # rank 1 is the slow one for the first value, rank 0 for the second
        local = [2.0 + rank, 5.0 - rank]
        got = bench.max_over_ranks(local)
        dist.barrier()
        out.put((rank, got, bench.whole_job_rate(2048, world, got[0])))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, rate in res:
        assert got == [3.0, 5.0]
        assert rate == pytest.approx(2 * 2048 / 3e-3)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert bench.whole_job_rate(100, 1, 2.0) == pytest.approx(50000.0)


def _shard_rank(rank, world, port, out):
    """One rank of a slot-range-sharded pool: oracle partials of its own slots, then the
    exchange (all_gather over gloo) and the merge."""
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import numpy as np
    import torch
    import torch.distributed as dist
    from gen import small_random
    from oracle import attention as oatt
    from oracle import quant as oq
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = small_random(152, num_slots=800, rows=3, topk=120, pad_frac=0.05)
        kc, vc, ks, vs = oq.write_int8(wl.k_tokens, wl.v_tokens, wl.slot_mapping, wl.num_slots, "side")
        K, V = oatt.int8_side_pool_fp64(kc, ks), oatt.int8_side_pool_fp64(vc, vs)
        lo, hi = rank * 800 // world, (rank + 1) * 800 // world
        mine = np.where((wl.topk >= lo) & (wl.topk < hi), wl.topk, -1)
        o, lse = oatt.gather_attention(wl.q, K, V, mine, wl.softmax_scale)
        o_all = [torch.empty(o.shape, dtype=torch.float64) for _ in range(world)]
        l_all = [torch.empty(lse.shape, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(o_all, torch.from_numpy(o))
        dist.all_gather(l_all, torch.from_numpy(lse))
        o_part = np.stack([t.numpy() for t in o_all], axis=1)
        l_part = np.stack([t.numpy() for t in l_all], axis=1)
        mo, ml = oatt.merge_splits(o_part, l_part)
        ro, rl = oatt.gather_attention(wl.q, K, V, wl.topk, wl.softmax_scale)
        out.put((rank, float(np.max(np.abs(mo - ro))), float(np.max(np.abs(ml - rl)))))
    finally:
        dist.destroy_process_group()


def test_slot_range_sharding_exchange_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, err_o, err_l in res:
        assert err_o < 1e-12 and err_l < 1e-12

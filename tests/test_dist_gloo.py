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

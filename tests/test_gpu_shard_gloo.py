"""A slot-range-sharded pool across two gloo ranks, with the library's own partials (GPU).

Each rank is a separate process with its own CUDA context on the one GPU of this machine. A rank
holds only its own slot range, written with the library at local ids, and attends the rows'
global entries in shard mode (qsa_gather_attn_ex with slot_lo: other ranks' entries are
skipped; a normalised partial and its lse come out), and the ranks exchange those
partials with one all_gather over gloo (host tensors). Every rank then merges the gathered
partials with qsa_splitk_merge and must match the oracle's unsharded attention. The ranks'
kernels never wait on one another: the only exchange is the host collective between launches.
("[Model][SM70][FP8] Add calibrated E4M3 QSA KV cache" §Implementation scope: split-K
workspace and merge.)
"""

import os
import socket

import pytest
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, fmt, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    sys.path.insert(0, os.path.join(root, "tests"))
    import numpy as np
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import quantized_kv_cache_write_gb300 as q
        from gen import small_random
        from harness import GpuPool, OraclePool, act_dev
        torch.cuda.set_device(0)
        import dataclasses
        wl = small_random(153, num_slots=5000, rows=7, topk=600, pad_frac=0.05, outlier_frac=0.02)
        R, Hq, D, S = wl.rows, wl.num_q_heads, wl.head_dim, wl.num_slots
        lo, hi = rank * S // world, (rank + 1) * S // world
        # this rank holds only its own slots, at local ids; the rows keep their global ids
        sm = wl.slot_mapping
        local = dataclasses.replace(wl, num_slots=hi - lo, slot_mapping=np.where((sm >= lo) & (sm < hi), sm - lo, -1))
        gp = GpuPool(local, fmt)
        o = torch.empty((R, Hq, D), dtype=torch.float32, device="cuda")
        lse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        q.qsa_gather_attn_ex(act_dev(wl.q), gp.code, gp.k_cache, gp.v_cache,
                             torch.from_numpy(np.ascontiguousarray(wl.topk, dtype=np.int32)).cuda(), wl.softmax_scale,
                             num_slots=hi - lo, k_scale_tok=gp.k_scale_tok, v_scale_tok=gp.v_scale_tok,
                             k_scale_layer=float(gp.k_scale_layer), v_scale_layer=float(gp.v_scale_layer),
                             out=o, lse=lse, dev_status=status, slot_lo=lo)
        torch.cuda.synchronize()
        assert status.item() == 0
        # the exchange: every rank's (o, lse) partial, gathered on the host
        o_all = [torch.empty((R, Hq, D), dtype=torch.float32) for _ in range(world)]
        l_all = [torch.empty((R, Hq), dtype=torch.float32) for _ in range(world)]
        dist.all_gather(o_all, o.cpu())
        dist.all_gather(l_all, lse.cpu())
        o_part = torch.stack(o_all, dim=1).contiguous().cuda()
        l_part = torch.stack(l_all, dim=1).contiguous().cuda()
        merged = torch.empty((R, Hq, D), dtype=torch.float32, device="cuda")
        mlse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
        q.qsa_splitk_merge(o_part, l_part, merged, mlse)  # the V scales are inside the partials
        torch.cuda.synchronize()
        ro, rl = OraclePool(wl, fmt).attend(wl)
        m = merged.cpu().numpy()
        ml = mlse.cpu().numpy()
        ok = bool(np.all(np.abs(m - ro) <= 5e-5 + 1e-3 * np.abs(ro)) and
                  np.all(np.abs(ml - rl) <= 5e-5 + 1e-3 * np.abs(rl)))
        out.put((rank, ok, float(np.max(np.abs(m - ro)))))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("fmt", ["int8_side", "e4m3"])
def test_two_gloo_ranks_exchange_library_partials(fmt):
    ctx = mp.get_context("spawn")
    res_q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, fmt, res_q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [res_q.get(timeout=600) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, ok, err in res:
        assert ok, (rank, err)

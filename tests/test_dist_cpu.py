"""The N > 1 path on the CPU: two gloo ranks (world size 2, 127.0.0.1).

Token rows are independent, so the benchmark shards them across GPUs with no
data-path collective: every rank draws and reduces its own rows, and only the
timing meets (a barrier and a max over ranks).  These tests run that host
logic with gloo and check the property that makes it valid: the op on a shard
of rows equals the same rows of the op on the whole batch (oracle, fp64).
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    try:
        import bench
        import oracle
        from gen import CONFIGS, make_inputs, problem_bytes
        from tests._util import oracle_args
        dist.init_process_group("gloo", rank=rank, world_size=world)
        oracle.set_num_threads(1)
        cfg = CONFIGS["tiny"]
        # 1) each rank draws its own shard: the shards differ
        mine = make_inputs(cfg, 4, seed=bench.rank_seed(cfg.index, 4, rank))
        digests = [None] * world
        dist.all_gather_object(digests, mine["residual"].float().sum().item())
        assert len(set(digests)) == world
        # 2) the timing reduction takes the slowest rank
        t = 1.5 + rank
        got = bench.max_over_ranks(t, world, "cpu")
        assert got == 1.5 + world - 1
        # 3) the reported value is all ranks' bytes over that time
        b = problem_bytes(cfg.R, cfg.K, cfg.H, 4)
        v = bench.aggregate_gbs(b, 10, got, world)
        assert abs(v - world * b * 10 / (got * 1e-3) / 1e9) < 1e-9
        # 4) sharding rows gives the same rows as the whole batch
        whole = make_inputs(cfg, 8, seed=123)
        rows = slice(4 * rank, 4 * rank + 4)
        K = cfg.K
        sub = dict(whole)
        sub["T"] = 4
        gathered = whole["perm"][rows].reshape(-1).long()
        sub["E"] = [e[gathered] for e in whole["E"]]
        sub["perm"] = torch.arange(4 * K, dtype=torch.int32).view(4, K)
        sub["w"] = whole["w"][rows]
        sub["S"] = [s[rows] for s in whole["S"]]
        sub["residual"] = whole["residual"][rows]
        a = oracle_args(sub)
        part = oracle.ar_finalize_rmsnorm_ref(a["E"], a["perm"], a["w"], a["S"], a["residual"],
                                              a["gamma"], a["weight_bias"], a["eps"])["out"]
        parts = [None] * world
        dist.all_gather_object(parts, part)
        a = oracle_args(whole)
        full = oracle.ar_finalize_rmsnorm_ref(a["E"], a["perm"], a["w"], a["S"], a["residual"],
                                              a["gamma"], a["weight_bias"], a["eps"])["out"]
        assert np.array_equal(np.concatenate(parts), full)
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, "ok"))
    except Exception as e:  # report, do not hang the other rank
        q.put((rank, repr(e)))
        raise


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    for p in procs:
        if p.is_alive():
            p.kill()
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: "ok", 1: "ok"}, res

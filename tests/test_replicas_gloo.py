"""Multi-rank host logic on CPU (gloo, world size 2, no GPU).

bench.py runs one independent replica per GPU (rows and batches of the
indexer are independent; no collective touches the data path) and reduces
only timings and work counts across ranks.  The same independence is what
row-sharded selection relies on ("DSV4: Add indexer_save_selection and
indexer_sharded_topk", Description): each rank selects its own slice of query
rows, positioned by q_start, and the gathered slices equal the full run.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    from oracle import csa_oracle as O

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        res = {}
        res["max"] = bench.max_over_ranks(float(rank + 1) * 1.5, dist)
        res["sum"] = bench.sum_over_ranks(float(rank + 1), dist)
        bench.barrier(dist)
        # row-sharded selection: rank r owns rows [r*S/world, (r+1)*S/world)
        rng = np.random.default_rng(0)  # same problem on every rank
        B, H, S, D, W, r, k = 2, 3, 40, 8, 10, 4, 4
        q = rng.standard_normal((B, H, S, D))
        kk = rng.standard_normal((B, W, D))
        w = rng.standard_normal((B, S, H))
        s0, s1 = rank * S // world, (rank + 1) * S // world
        start = np.full(B, s0, dtype=np.int64)
        _, idx = O.index_topk(q[:, :, s0:s1], kk, w[:, s0:s1], 0.3, r, k, q_start=start)
        parts = [torch.zeros(B, S // world, k, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(parts, torch.from_numpy(idx))
        _, full = O.index_topk(q, kk, w, 0.3, r, k)
        res["shards_equal_full"] = bool(np.array_equal(torch.cat(parts, dim=1).numpy(), full))
        out_q.put((rank, res))
    finally:
        dist.destroy_process_group()


def test_two_rank_reductions_and_row_shards():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in range(2):
        assert results[rank]["max"] == 3.0
        assert results[rank]["sum"] == 3.0
        assert results[rank]["shards_equal_full"]


def test_replica_inputs_differ_by_rank():
    from csa_inputs import WORKLOADS, make_inputs
    wl = WORKLOADS["tiny"]
    a = make_inputs(wl.with_(seed=wl.seed + 0))
    b = make_inputs(wl.with_(seed=wl.seed + 1))
    assert not torch.equal(a.q, b.q)


def test_row_shard_cut_points():
    """Row ranges cover every row once, inner cuts on 4-row blocks, and the
    visible-entry work of the shards is balanced (later rows see more)."""
    from sparse_attention_indexer_csa_gb300.shard import row_shards, visible_entries

    for S, W, r, n, start in [(16384, 4096, 4, 2, 0), (16384, 4096, 4, 8, 0), (4096, 1024, 4, 3, 0),
                              (600, 1024, 4, 2, 2000), (10, 4, 4, 4, 0), (7, 100, 1, 2, 0)]:
        cuts = row_shards(S, W, r, n, start)
        assert len(cuts) == n and cuts[0][0] == 0 and cuts[-1][1] == S
        assert all(cuts[i][1] == cuts[i + 1][0] for i in range(n - 1))
        assert all(b <= e for b, e in cuts)
        assert all(e % 4 == 0 for _, e in cuts[:-1])
        work = [sum(visible_entries(s, W, r, start) for s in range(b, e)) for b, e in cuts]
        if S >= 1024:
            # a 4-row block of the heaviest rows is the granularity of the balance
            assert max(work) - min(work) <= 2 * 4 * W, (S, n, work)

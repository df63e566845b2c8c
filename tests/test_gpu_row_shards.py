"""Row-sharded selection on the CUDA path (GPU): two ranks (processes, gloo
for the one gather) each run their own contiguous range of query rows of
one problem through the library, positioned by q_start, on the same GPU.
Their kernels never wait on one another.  The gathered indices must equal
one call over all rows bit for bit ("DSV4: Add indexer_save_selection and
indexer_sharded_topk", Description: the sharded top-k leaves the selection
unchanged), and sampled rows must match the oracle.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu

WORLD = 2


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _case(name):
    from csa_inputs import WORKLOADS
    if name == "prefill":
        return WORKLOADS["prefill_4k"].with_(seed=21)
    if name == "packed":
        return WORKLOADS["packed_8k"].with_(B=2, S=1024, W=256, top_k=40, seed=1)
    return WORKLOADS["prefill_4k"].with_(B=3, S=600, W=1024, top_k=100, q_start=2000, seed=22)


def _worker(rank, port, name, out_q):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import sparse_attention_indexer_csa_gb300 as csa
    from csa_inputs import make_inputs
    from sparse_attention_indexer_csa_gb300.shard import row_shards

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=WORLD)
    try:
        torch.cuda.set_device(0)
        csa.load()
        wl = _case(name)
        inp = make_inputs(wl)  # the same problem on every rank
        s0, s1 = row_shards(wl.S, wl.W, wl.compress_rate, WORLD, wl.q_start or 0)[rank]
        base = inp.q_start if inp.q_start is not None else torch.zeros(wl.B, dtype=torch.int64)
        g = lambda t: None if t is None else t.cuda().contiguous()  # noqa: E731
        idx = csa.index_fused(g(inp.q[:, :, s0:s1]), g(inp.k), g(inp.w[:, s0:s1]), wl.scale, wl.compress_rate,
                              wl.top_k, None if inp.q_seg is None else g(inp.q_seg[:, s0:s1]), g(inp.kv_seg),
                              g(base + s0))
        torch.cuda.synchronize()
        assert csa.device_status() == csa.CSA_OK
        rows = torch.tensor([s1 - s0])
        all_rows = [torch.zeros(1, dtype=torch.int64) for _ in range(WORLD)]
        dist.all_gather(all_rows, rows)
        maxr = int(max(r.item() for r in all_rows))
        pad = torch.full((wl.B, maxr, wl.top_k), -2, dtype=torch.int32)
        pad[:, :s1 - s0] = idx.cpu()
        parts = [torch.empty_like(pad) for _ in range(WORLD)]
        dist.all_gather(parts, pad)
        res = {}
        if rank == 0:
            shards = row_shards(wl.S, wl.W, wl.compress_rate, WORLD, wl.q_start or 0)
            got = torch.cat([parts[r][:, :e - b] for r, (b, e) in enumerate(shards)], dim=1)
            full = csa.index_fused(g(inp.q), g(inp.k), g(inp.w), wl.scale, wl.compress_rate, wl.top_k,
                                   g(inp.q_seg), g(inp.kv_seg), g(inp.q_start))
            res["shards"] = shards
            res["equal_full"] = bool(torch.equal(got, full.cpu()))
            res["idx"] = got.numpy()
        out_q.put((rank, res))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name", ["prefill", "packed", "offset"])
def test_row_shards_equal_one_full_call(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from csa_inputs import make_inputs
    from oracle import csa_oracle as O
    from parity import check_select_vs_oracle, oracle_scores

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, name, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=600) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    r0 = results[0]
    (a0, a1), (b0, b1) = r0["shards"]
    assert a0 == 0 and a1 == b0 and b1 == _case(name).S and a1 % 4 == 0
    assert r0["equal_full"], "gathered row shards differ from one call over all rows"
    # sampled rows of both shards against the oracle's own scores
    wl = _case(name)
    inp = make_inputs(wl)
    rows = np.unique(np.clip(np.array([0, 1, a1 - 2, a1 - 1, a1, a1 + 1, wl.S // 3, wl.S - 2, wl.S - 1]), 0,
                             wl.S - 1))
    ref = oracle_scores(inp, rows=rows)
    check_select_vs_oracle(ref, r0["idx"][:, rows], wl.top_k)
    assert O.select_topk(ref, wl.top_k).shape == r0["idx"][:, rows].shape

"""Host-side checks of bench.py's accounting (no GPU): the work counts
behind every reported TFLOP/s and rows/s, the L2 rule, and the algorithmic
bytes of the decode roofline."""
import numpy as np
import pytest
import torch

import bench
from csa_inputs import WORKLOADS, Inputs, make_inputs


def _shape_only(wl, q_start=None):
    """Inputs carrying only what the work count reads (no tensors drawn)."""
    qs = None if q_start is None else torch.tensor(q_start, dtype=torch.int64)
    return Inputs(wl, None, None, None, None, None, qs)


def _brute_visible(wl, q_start=None, q_seg=None, kv_seg=None):
    """Visible entries per row by the definition, one entry at a time."""
    v = np.zeros((wl.B, wl.S), dtype=np.int64)
    for b in range(wl.B):
        qs = 0 if q_start is None else int(q_start[b])
        for s in range(wl.S):
            n = 0
            for t in range(wl.W):
                if t * wl.compress_rate + wl.compress_rate - 1 <= qs + s and (
                        q_seg is None or q_seg[b, s] == kv_seg[b, t]):
                    n += 1
            v[b, s] = n
    return v


# per-config work of the contract table: (visible pairs, rows above top_k)
TABLE = {"tiny": (8128, 189), "prefill_4k": (2096128, 2045), "prefill_16k": (67100672, 16378),
         "decode_32k": (2097152, 64)}


@pytest.mark.parametrize("name", sorted(TABLE))
def test_work_matches_the_contract_table(name):
    wl = WORKLOADS[name]
    wk = bench.work(_shape_only(wl, None if wl.q_start is None else [wl.q_start] * wl.B))
    pairs, nontrivial = TABLE[name]
    assert wk["pairs"] == pairs
    assert wk["nontrivial_rows"] == nontrivial
    assert wk["flops"] == 2 * wl.H * wl.D * pairs
    assert wk["rows"] == wl.B * wl.S


def test_prefill_16k_flops():
    wk = bench.work(_shape_only(WORKLOADS["prefill_16k"]))
    assert abs(wk["flops"] / 1e12 - 1.0994) < 5e-4
    assert abs(wk["flops_nontrivial"] / 1e12 - 0.824) < 5e-3


@pytest.mark.parametrize("case", [dict(B=2, S=37, W=9, compress_rate=4, q_start=[0, 5]),
                                  dict(B=1, S=40, W=13, compress_rate=3, q_start=[-7]),
                                  dict(B=2, S=30, W=30, compress_rate=1, q_start=None)])
def test_visible_counts_by_brute_force(case):
    qs = case.pop("q_start")
    wl = WORKLOADS["tiny"].with_(**case)
    v = bench.visible_counts(_shape_only(wl, qs))
    assert np.array_equal(v, _brute_visible(wl, qs))


def test_visible_counts_with_segments_by_brute_force():
    wl = WORKLOADS["packed_8k"].with_(B=2, S=64, W=16, H=4, D=32, top_k=4, seed=3)
    inp = make_inputs(wl)
    v = bench.visible_counts(inp)
    assert np.array_equal(v, _brute_visible(wl, None, inp.q_seg.numpy(), inp.kv_seg.numpy()))


def test_l2_rule():
    for name in ("tiny", "prefill_4k"):
        assert bench.needs_l2_flush(WORKLOADS[name])
        assert bench.config_dict(WORKLOADS[name], 1)["l2"].startswith("flushed")
    for name in ("prefill_16k", "packed_8k", "decode_32k", "prefill_64k"):
        assert not bench.needs_l2_flush(WORKLOADS[name])
        assert bench.config_dict(WORKLOADS[name], 1)["l2"].startswith("no flush")
    assert bench.input_bytes(WORKLOADS["prefill_16k"]) == (2 * 64 * 16384 * 128 * 2 + 2 * 4096 * 128 * 2
                                                          + 2 * 16384 * 64 * 2)


def test_decode_bytes():
    wl = WORKLOADS["decode_32k"]
    k = 64 * 32768 * 128 * 2
    q = 64 * 64 * 128 * 2
    w = 64 * 64 * 2
    scores = 2 * 64 * 32768 * 4  # written by the score pass, read back by the selection
    idx = 64 * 2048 * 4
    assert bench.decode_bytes(wl) == k + q + w + scores + idx

"""Shared helpers of the GPU parity tests: run the library through its C ABI
on seeded inputs and compare with the CPU oracle.

Tolerance (scores): |gpu - oracle| <= 2e-3 * max_t |oracle[b,s,t]| over the
row's visible entries; masked entries must be -inf on both sides.
Selection: (1) the oracle's selector run on the GPU's own fp32 scores must
reproduce the GPU indices exactly; (2) against the oracle's fp64 scores the
index sets may differ only in entries within the row tolerance of the
oracle's k-th value, and the -1 padding counts must match exactly.
"""
from __future__ import annotations

import numpy as np
import torch

import sparse_attention_indexer_csa_gb300 as csa
from csa_inputs import Inputs
from oracle import csa_oracle as O

TOL = 2e-3


def np_inputs(inp: Inputs):
    f = lambda t: None if t is None else t.double().numpy()  # noqa: E731
    i = lambda t: None if t is None else t.numpy()  # noqa: E731
    return dict(q=f(inp.q), k=f(inp.k), w=f(inp.w), q_start=i(inp.q_start), q_seg=i(inp.q_seg),
                kv_seg=i(inp.kv_seg))


def to_dev(inp: Inputs, dev="cuda"):
    g = lambda t: None if t is None else t.to(dev).contiguous()  # noqa: E731
    return dict(q=g(inp.q), k=g(inp.k), w=g(inp.w), q_start=g(inp.q_start), q_seg=g(inp.q_seg),
                kv_seg=g(inp.kv_seg))


def oracle_scores(inp: Inputs, rows=None):
    a = np_inputs(inp)
    wl = inp.wl
    return O.index_scores(a["q"], a["k"], a["w"], wl.scale, wl.compress_rate, a["q_start"], a["q_seg"],
                          a["kv_seg"], rows=rows)


def gpu_scores(inp: Inputs, d=None):
    d = d or to_dev(inp)
    wl = inp.wl
    return csa.index_score(d["q"], d["k"], d["w"], wl.scale, wl.compress_rate, d["q_seg"], d["kv_seg"],
                           d["q_start"])


def gpu_fused(inp: Inputs, d=None, dbg=False):
    d = d or to_dev(inp)
    wl = inp.wl
    sd = None
    if dbg:
        sd = torch.full((wl.B, wl.S, wl.W), float("nan"), dtype=torch.float32, device=d["q"].device)
    idx = csa.index_fused(d["q"], d["k"], d["w"], wl.scale, wl.compress_rate, wl.top_k, d["q_seg"],
                          d["kv_seg"], d["q_start"], scores_dbg=sd)
    return idx, sd


def assert_status_ok():
    torch.cuda.synchronize()
    st = csa.device_status()
    assert st == csa.CSA_OK, f"device status word: {st}"


def check_scores(g: np.ndarray, ref: np.ndarray):
    """Element-wise score parity on the rows given (same shape)."""
    fin = np.isfinite(ref)
    assert np.array_equal(fin, np.isfinite(g)), "mask differs (finite vs -inf)"
    assert np.all(g[~fin] == -np.inf) and np.all(ref[~fin] == -np.inf)
    rowmax = np.max(np.where(fin, np.abs(ref), 0.0), axis=-1, keepdims=True)
    err = np.abs(np.where(fin, g, 0.0) - np.where(fin, ref, 0.0))
    bad = err > TOL * rowmax
    assert not bad.any(), (f"{int(bad.sum())} scores outside tolerance; worst rel "
                           f"{float((err / np.maximum(rowmax, 1e-300)).max()):.3e}")
    return float((err / np.maximum(rowmax, 1e-300)).max())


def select_rows_chunked(sc: np.ndarray, k: int, chunk: int = 4096):
    flat = sc.reshape(-1, sc.shape[-1])
    out = np.empty((flat.shape[0], k), dtype=np.int64)
    for i in range(0, flat.shape[0], chunk):
        out[i:i + chunk] = O.select_topk(flat[i:i + chunk].astype(np.float64), k)
    return out.reshape(*sc.shape[:-1], k)


def check_select_exact(g_scores: np.ndarray, g_idx: np.ndarray, k: int):
    """The oracle's selector on the GPU's fp32 scores gives the GPU's indices."""
    ref = select_rows_chunked(g_scores, k)
    mism = np.nonzero(np.any(ref != g_idx, axis=-1).reshape(-1))[0]
    assert mism.size == 0, f"{mism.size} rows differ from the oracle selector, first row {mism[0]}"


def check_select_vs_oracle(ref_sc: np.ndarray, g_idx: np.ndarray, k: int):
    """Index sets equal except for entries within tolerance of the k-th value."""
    ref_idx = O.select_topk(ref_sc, k)
    flat_sc = ref_sc.reshape(-1, ref_sc.shape[-1])
    fi = g_idx.reshape(-1, k)
    fr = ref_idx.reshape(-1, k)
    for r in range(flat_sc.shape[0]):
        row = flat_sc[r]
        vis = np.isfinite(row)
        assert (fi[r] < 0).sum() == (fr[r] < 0).sum(), f"row {r}: padding count differs"
        nvis = int(vis.sum())
        if nvis <= k:
            assert np.array_equal(fi[r], fr[r]), f"row {r}: visible set differs"
            continue
        tol = TOL * np.max(np.abs(row[vis]))
        vk = np.sort(row[vis])[::-1][k - 1]
        boundary = vis & (np.abs(row - vk) <= tol)
        gs = set(int(t) for t in fi[r] if t >= 0)
        rs = set(int(t) for t in fr[r] if t >= 0)
        for t in rs - gs:
            assert boundary[t], f"row {r}: oracle-selected entry {t} missing and not at the boundary"
        for t in gs - rs:
            assert boundary[t], f"row {r}: entry {t} selected but not at the boundary"
        assert all(vis[t] for t in gs), f"row {r}: masked entry selected"

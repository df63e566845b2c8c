"""Backward of the score step on the GPU (csa_index_backward) against the
oracle's ``index_scores_vjp``.

Tolerances follow from the arithmetic of the GPU path:
* P = gm * w * scale * [x > 0] is rounded to bf16 before the dq / dk GEMMs
  (8 significant bits: at most 2^-8 relative per term); the GEMMs accumulate
  in fp32.  So |dq - dq_ref| <= 2^-7 * (|P| @ |k|) per element, and likewise
  for dk with |P|^T @ |q| summed over heads (a factor 2 above the rounding
  bound).
* x = q.k comes from the tensor cores' fp32 accumulation of bf16 products
  (error far below 1e-4 * |q|.|k|): where |x| is within that margin the ReLU
  gate may differ between fp32 and fp64, so those entries' full terms are
  allowed.
* dw is accumulated in fp32 from those fp32 logits: 1e-4 of sum |gm| * scale
  * |q|.|k| (the same envelope of the logits' error).
Full-size problems are checked on sampled rows (dq, dw) and, for dk, by
Euler's identity: the score is degree-1 homogeneous in q, k and w, so
sum(q*dq), sum(k*dk) and sum(w*dw) all equal sum(g * score).
"""
import json
import os

import numpy as np
import pytest
import torch

import sparse_attention_indexer_csa_gb300 as csa
from csa_inputs import WORKLOADS, Workload, make_inputs, to_f64
from oracle import csa_oracle as O

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    csa.load()


def _cot(B, S, W, seed):
    gen = torch.Generator().manual_seed(seed)
    return torch.randn(B, S, W, generator=gen, dtype=torch.float32)


def _bounds(q, k, w, scale, r, g, q_start=None, q_seg=None, kv_seg=None, rows=None):
    """Per-element error bounds (dq [B,H,R,D], dk [B,W,D] or None, dw [B,R,H]) for rows `rows`."""
    B, H, S, D = q.shape
    W = k.shape[1]
    rows = np.arange(S) if rows is None else np.asarray(rows)
    c = O.scale_value(scale)
    vis = O.visibility(B, S, W, r, q_start, q_seg, kv_seg, rows)
    gm = np.where(vis, g[:, rows], 0.0)
    bdq = np.zeros((B, H, len(rows), D))
    bdw = np.zeros((B, len(rows), H))
    bdk = np.zeros((B, W, D)) if len(rows) == S else None
    for b in range(B):
        for h in range(H):
            qb = q[b, h][rows]
            x = qb @ k[b].T
            mag = np.abs(qb) @ np.abs(k[b]).T             # |q|.|k| per pair
            amb = np.abs(x) <= 1e-4 * mag                  # ReLU gate may differ in fp32
            pabs = np.abs(gm[b]) * abs(w[b, rows, h])[:, None] * c
            term = 2.0 ** -7 * pabs * (x > 0) + pabs * amb
            bdq[b, h] = term @ np.abs(k[b])
            bdw[b, :, h] = 1e-4 * (np.abs(gm[b]) * c * mag).sum(axis=1)
            if bdk is not None:
                bdk[b] += term.T @ np.abs(qb)
    floor = 1e-7
    return bdq + floor, (None if bdk is None else bdk + floor), bdw + floor


def _dev(inp):
    f = lambda t: None if t is None else t.cuda().contiguous()  # noqa: E731
    return f(inp.q), f(inp.k), f(inp.w), f(inp.q_seg), f(inp.kv_seg), f(inp.q_start)


def _np(t):
    return None if t is None else t.numpy()


def _run_and_check(inp, seed):
    wl = inp.wl
    q, k, w, qs, ks, st = _dev(inp)
    g = _cot(wl.B, wl.S, wl.W, seed)
    dq, dk, dw = csa.index_backward(q, k, w, wl.scale, wl.compress_rate, g.cuda(), qs, ks, st)
    torch.cuda.synchronize()
    assert csa.device_status() == csa.CSA_OK
    Q, K, Wt = to_f64(inp.q), to_f64(inp.k), to_f64(inp.w)
    G = g.double().numpy()
    args = (_np(inp.q_start), _np(inp.q_seg), _np(inp.kv_seg))
    rq, rk, rw = O.index_scores_vjp(Q, K, Wt, wl.scale, wl.compress_rate, G, *args)
    bq, bk, bw = _bounds(Q, K, Wt, wl.scale, wl.compress_rate, G, *args)
    for name, got, ref, bd in (("dq", dq, rq, bq), ("dk", dk, rk, bk), ("dw", dw, rw, bw)):
        err = np.abs(got.double().cpu().numpy() - ref)
        bad = err > bd
        assert not bad.any(), f"{name}: {int(bad.sum())} elements outside bound; worst {float((err / bd).max()):.2f}x"


def test_hand_example_exact_in_64_heads():
    """The golden 2-head / 2-dim gradient example, zero-padded to 64 heads and
    128 dims: every value is exact in bf16 / fp32, so the GPU must match."""
    with open(os.path.join(GOLDEN, "hand_example.json")) as f:
        gj = json.load(f)
    S, W = gj["S"], gj["W"]
    q = torch.zeros(1, 64, S, 128)
    k = torch.zeros(1, W, 128)
    w = torch.zeros(1, S, 64)
    q[0, :2, :, :2] = torch.tensor(gj["q"], dtype=torch.float32)
    k[0, :, :2] = torch.tensor(gj["k"], dtype=torch.float32)
    w[0, :, :2] = torch.tensor(gj["w"], dtype=torch.float32)
    g = torch.zeros(1, S, W)
    for s_, t_, v in gj["backward_example"]["g_entries"]:
        g[0, s_, t_] = v
    dq, dk, dw = csa.index_backward(q.bfloat16().cuda(), k.bfloat16().cuda(), w.bfloat16().cuda(), gj["scale"],
                                    gj["compress_rate"], g.cuda())
    torch.cuda.synchronize()
    edq, edk, edw = torch.zeros_like(dq), torch.zeros_like(dk), torch.zeros_like(dw)
    for h, s_, d, v in gj["backward_example"]["expected_dq_nonzero"]:
        edq[0, h, s_, d] = v
    for t_, d, v in gj["backward_example"]["expected_dk_nonzero"]:
        edk[0, t_, d] = v
    for s_, h, v in gj["backward_example"]["expected_dw_nonzero"]:
        edw[0, s_, h] = v
    assert torch.equal(dq, edq) and torch.equal(dk, edk) and torch.equal(dw, edw)


@pytest.mark.parametrize("case", [
    dict(B=2, S=301, W=100, seed=1),                          # odd rows (last pair half empty), W % 128 != 0
    dict(B=1, S=256, W=300, seed=2, w_dtype="f32"),
    dict(B=2, S=200, W=64, seed=3, docs=(2, 4)),             # packed documents: segment mask
    dict(B=2, S=2048, W=512, seed=11, docs=(3, 8)),          # documents over several tiles: tiles and pairs skipped
    dict(B=2, S=1536, W=900, seed=12, docs=(2, 5), q_start=2000),  # documents with offset rows
    dict(B=2, S=40, W=700, seed=4, q_start=600),             # offset rows: every chunk spans all entries
    dict(B=3, S=1, W=1000, seed=8, q_start=5000),            # one row per sequence (decode shape)
    dict(B=1, S=100, W=6000, seed=9, q_start=30000),         # rows longer than 4096 entries (47 tiles)
])
def test_backward_matches_oracle(case):
    case = dict(case)
    seed = case.pop("seed")
    base = WORKLOADS["prefill_4k"]
    wl = base.with_(seed=seed, top_k=16, **case)
    _run_and_check(make_inputs(wl), seed)


def test_backward_sequence_major_q():
    # q [B,S,H,D]: dq comes back in the same layout and equals the head-major
    # result within the same bounds (the oracle works on the head-major view)
    wl = WORKLOADS["prefill_4k"].with_(B=2, S=2100, W=600, seed=10, top_k=16)
    inp = make_inputs(wl)
    q, k, w, qs, ks, st = _dev(inp)
    qsm = q.transpose(1, 2).contiguous()
    g = _cot(wl.B, wl.S, wl.W, 10)
    dq, dk, dw = csa.index_backward(qsm, k, w, wl.scale, wl.compress_rate, g.cuda(), q_layout=csa.CSA_Q_SEQ_MAJOR)
    torch.cuda.synchronize()
    assert csa.device_status() == csa.CSA_OK
    assert dq.shape == qsm.shape
    Q, K, Wt = to_f64(inp.q), to_f64(inp.k), to_f64(inp.w)
    G = g.double().numpy()
    rq, rk, rw = O.index_scores_vjp(Q, K, Wt, wl.scale, wl.compress_rate, G)
    bq, bk, bw = _bounds(Q, K, Wt, wl.scale, wl.compress_rate, G)
    got_dq = dq.transpose(1, 2).double().cpu().numpy()
    for name, got, ref, bd in (("dq", got_dq, rq, bq), ("dk", dk.double().cpu().numpy(), rk, bk),
                               ("dw", dw.double().cpu().numpy(), rw, bw)):
        bad = np.abs(got - ref) > bd
        assert not bad.any(), f"{name}: {int(bad.sum())} elements outside bound"


@pytest.mark.parametrize("S", [2100, 8300])
def test_backward_several_chunks(S):
    # 2100 rows: one chunk, GEMM sub-blocks of 2048 and 52 rows with growing
    # ranges; 8300 rows: a chunk of 8192 rows (four sub-blocks) and one of 108
    wl = WORKLOADS["prefill_4k"].with_(B=1, S=S, W=600, seed=5, top_k=16)
    _run_and_check(make_inputs(wl), 5)


def test_backward_no_visible_rows():
    # compress_rate above every position + 1: nothing is visible, all gradients zero
    wl = WORKLOADS["prefill_4k"].with_(B=1, S=6, W=8, compress_rate=16, seed=6, top_k=4)
    inp = make_inputs(wl)
    q, k, w, qs, ks, st = _dev(inp)
    dq, dk, dw = csa.index_backward(q, k, w, wl.scale, wl.compress_rate, _cot(1, 6, 8, 6).cuda())
    torch.cuda.synchronize()
    assert not dq.any() and not dk.any() and not dw.any()


def test_backward_full_size_sampled_rows_and_euler_identity():
    wl = WORKLOADS["prefill_16k"]
    inp = make_inputs(wl)
    q, k, w, qs, ks, st = _dev(inp)
    g = _cot(wl.B, wl.S, wl.W, 7)
    gd = g.cuda()
    dq, dk, dw = csa.index_backward(q, k, w, wl.scale, wl.compress_rate, gd)
    sc = csa.index_score(q, k, w, wl.scale, wl.compress_rate)
    torch.cuda.synchronize()
    assert csa.device_status() == csa.CSA_OK
    # Euler: all three equal sum(g * score) over visible entries
    vis = torch.isfinite(sc)
    L = float((torch.where(vis, gd, 0.0).double() * torch.where(vis, sc, 0.0).double()).sum())
    sq = float((q.double() * dq.double()).sum())
    sk = float((k.double() * dk.double()).sum())
    sw = float((w.double() * dw.double()).sum())
    # error scale: sum |g| * sum_h |w| ReLU(scale x) = sum |P| |x|, the score
    # with |w|; bf16 rounding of P moves sum(q*dq) and sum(k*dk) by at most
    # 2^-8 of it (bound taken with a factor 2); sum(w*dw) and sum(g*score)
    # differ by the logits' fp32 error (two products, different orders)
    sa = csa.index_score(q, k, w.abs(), wl.scale, wl.compress_rate)
    ref = float((torch.where(vis, gd.abs(), 0.0).double() * torch.where(vis, sa, 0.0).double()).sum())
    assert abs(sw - L) <= 1e-4 * ref
    assert abs(sq - L) <= 2.0 ** -7 * ref
    assert abs(sk - L) <= 2.0 ** -7 * ref
    # sampled rows of dq and dw against the oracle (the same bounds as above,
    # computed for these rows only)
    rows = np.array([0, 3, 4, 5, 777, 8191, 8192, 12345, 16383])
    Qr = inp.q[:, :, rows].double().numpy()
    K, Wt = to_f64(inp.k), to_f64(inp.w)
    G = g.double().numpy()
    c = O.scale_value(wl.scale)
    vism = O.visibility(wl.B, wl.S, wl.W, wl.compress_rate, rows=rows)
    gm = np.where(vism, G[:, rows], 0.0)
    dq_s = dq[:, :, rows].double().cpu().numpy()
    dw_s = dw[:, rows].double().cpu().numpy()
    for b in range(wl.B):
        for h in range(wl.H):
            x = Qr[b, h] @ K[b].T
            mag = np.abs(Qr[b, h]) @ np.abs(K[b]).T
            amb = np.abs(x) <= 1e-4 * mag
            pabs = np.abs(gm[b]) * np.abs(Wt[b, rows, h])[:, None] * c
            bq = (2.0 ** -7 * pabs * (x > 0) + pabs * amb) @ np.abs(K[b]) + 1e-7
            bw = 1e-4 * (np.abs(gm[b]) * c * mag).sum(axis=1) + 1e-7
            dx = gm[b] * Wt[b, rows, h][:, None] * c * (c * x > 0)
            assert (np.abs(dq_s[b, h] - dx @ K[b]) <= bq).all(), (b, h)
            assert (np.abs(dw_s[b, :, h] - (gm[b] * np.maximum(c * x, 0)).sum(axis=1)) <= bw).all(), (b, h)

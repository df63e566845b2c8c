"""Pins of the CPU oracle against things other than itself (no GPU).

Each test pins a part of ``oracle/csa_oracle.py`` with a hand-worked example,
a brute-force formulation, a special case that reduces to a textbook routine
or an invariant of the definition, chosen so that a dropped term, a wrong sign
or index, or a transposed operand fails at least one of them.
"""
import json
import os

import numpy as np
import pytest

from oracle import csa_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _hand():
    with open(os.path.join(GOLDEN, "hand_example.json")) as f:
        g = json.load(f)
    q = np.array(g["q"], dtype=np.float64)[None]          # [1,H,S,D]
    k = np.array(g["k"], dtype=np.float64)[None]          # [1,W,D]
    w = np.array(g["w"], dtype=np.float64)[None]          # [1,S,H]
    exp = np.array([[float(v) for v in row] for row in g["expected_scores"]])[None]
    return g, q, k, w, exp


def _rand_problem(rng, B, H, S, D, W, r, segs=False, start=None):
    q = rng.standard_normal((B, H, S, D))
    k = rng.standard_normal((B, W, D))
    w = rng.standard_normal((B, S, H))
    q_start = None if start is None else np.array(start, dtype=np.int64)
    q_seg = kv_seg = None
    if segs:
        q_seg = np.sort(rng.integers(0, 3, size=(B, S)), axis=1).astype(np.int32)
        kv_seg = rng.integers(0, 3, size=(B, W)).astype(np.int32)
    return q, k, w, q_start, q_seg, kv_seg


def _brute_select(row, top_k):
    """Selection by repeated arg-max with '>' (first occurrence wins ties)."""
    cand = [t for t, v in enumerate(row) if v > -np.inf]
    chosen = []
    for _ in range(min(top_k, len(cand))):
        best = None
        for t in cand:
            if t in chosen:
                continue
            if best is None or row[t] > row[best]:
                best = t
        chosen.append(best)
    return sorted(chosen) + [-1] * (top_k - len(chosen))


# --------------------------------------------------------------------------- hand example
def test_hand_example_scores_exact():
    g, q, k, w, exp = _hand()
    sc = O.index_scores(q, k, w, g["scale"], g["compress_rate"])
    assert np.array_equal(sc, exp)  # exact: every value is representable


def test_hand_example_topk():
    g, q, k, w, exp = _hand()
    _, idx = O.index_topk(q, k, w, g["scale"], g["compress_rate"], g["top_k"])
    assert idx[0].tolist() == g["expected_topk"]


def test_hand_example_brute_force():
    g, q, k, w, exp = _hand()
    sc = O.brute_force_scores(q, k, w, g["scale"], g["compress_rate"])
    assert np.array_equal(sc, exp)


def test_hand_example_padded_heads_and_dims():
    """Zero heads (q=0, w=0) and zero dims change nothing (a kernel pads both)."""
    g, q, k, w, exp = _hand()
    qp = np.zeros((1, 4, 8, 32)); qp[:, :2, :, :2] = q
    kp = np.zeros((1, 4, 32)); kp[:, :, :2] = k
    wp = np.zeros((1, 8, 4)); wp[:, :, :2] = w
    sc = O.index_scores(qp, kp, wp, g["scale"], g["compress_rate"])
    assert np.array_equal(sc, exp)


# --------------------------------------------------------------------------- brute force
@pytest.mark.parametrize("seed", range(6))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(100 + seed)
    H = [1, 2, 4][seed % 3]
    D = [2, 32][seed % 2]
    r = [1, 2, 3, 4][seed % 4]
    S = 24 if D == 32 else 48
    W = min(16, S // r + 2)
    segs = seed % 2 == 1
    start = [int(rng.integers(0, 9))] if seed >= 3 else None
    q, k, w, q_start, q_seg, kv_seg = _rand_problem(rng, 1, H, S, D, W, r, segs, start)
    scale = 0.37
    a = O.index_scores(q, k, w, scale, r, q_start, q_seg, kv_seg)
    b = O.brute_force_scores(q, k, w, scale, r, q_start, q_seg, kv_seg)
    assert np.array_equal(np.isinf(a), np.isinf(b))
    fin = np.isfinite(a)
    np.testing.assert_allclose(a[fin], b[fin], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", range(4))
def test_select_matches_repeated_argmax(seed):
    rng = np.random.default_rng(seed)
    sc = rng.integers(-3, 4, size=(20, 13)).astype(np.float64)  # many exact ties
    sc[rng.random(sc.shape) < 0.3] = -np.inf
    for top_k in (1, 4, 13, 20):
        got = O.select_topk(sc, top_k)
        for i in range(sc.shape[0]):
            assert got[i].tolist() == _brute_select(sc[i].tolist(), top_k)


def test_select_signed_zero_ties_by_value():
    row = np.array([[0.0, -0.0, 0.0, -1.0, -0.0]])
    assert O.select_topk(row, 2).tolist() == [[0, 1]]
    row = np.array([[-0.0, 0.0, -np.inf]])
    assert O.select_topk(row, 3).tolist() == [[0, 1, -1]]


def test_select_properties():
    rng = np.random.default_rng(7)
    sc = np.round(rng.standard_normal((64, 50)), 1)
    sc[rng.random(sc.shape) < 0.2] = -np.inf
    k = 17
    idx = O.select_topk(sc, k)
    for i in range(sc.shape[0]):
        vis = np.nonzero(sc[i] > -np.inf)[0]
        sel = [t for t in idx[i] if t >= 0]
        assert len(sel) == min(k, len(vis))
        assert sel == sorted(sel) and all(sc[i, t] > -np.inf for t in sel)
        uns = [t for t in vis if t not in sel]
        for a in sel:
            for b in uns:
                assert sc[i, a] > sc[i, b] or (sc[i, a] == sc[i, b] and a < b)


# --------------------------------------------------------------------------- special case
def test_single_head_unit_weight_is_relu_matmul_and_argsort():
    rng = np.random.default_rng(3)
    S, W, D = 40, 10, 8
    q = rng.standard_normal((1, 1, S, D))
    k = rng.standard_normal((1, W, D))
    w = np.ones((1, S, 1))
    start = np.array([10 * W])  # every entry visible
    sc = O.index_scores(q, k, w, 1.0, 1, q_start=start)
    ref = np.maximum(q[0, 0] @ k[0].T, 0.0)
    np.testing.assert_allclose(sc[0], ref, rtol=1e-13, atol=1e-13)
    idx = O.select_topk(sc, 4)[0]
    for s in range(S):
        expect = sorted(np.argsort(-ref[s], kind="stable")[:4].tolist())
        assert idx[s].tolist() == expect


def test_causal_threshold_values():
    # entry t covers tokens t*r .. t*r+r-1; visible once its last token <= pos
    r = 4
    for pos in range(40):
        n = sum(1 for t in range(20) if t * r + r - 1 <= pos)
        assert O.causal_threshold(pos, r) == n
    assert O.causal_threshold(131071, 4) == 32768


# --------------------------------------------------------------------------- invariants
def _prob(seed=0, segs=True, H=4, S=64, D=16, W=16, r=4, start=None):
    rng = np.random.default_rng(seed)
    return _rand_problem(rng, 2, H, S, D, W, r, segs, start)


def test_masked_never_selected():
    q, k, w, qs, qg, kg = _prob(1)
    sc, idx = O.index_topk(q, k, w, 0.25, 4, 8, qs, qg, kg)
    vis = O.visibility(2, 64, 16, 4, qs, qg, kg)
    for b in range(2):
        for s in range(64):
            for t in idx[b, s]:
                if t >= 0:
                    assert vis[b, s, t]


def test_zero_weights_zero_scores_lowest_indices():
    q, k, w, qs, qg, kg = _prob(2)
    w = np.zeros_like(w)
    sc, idx = O.index_topk(q, k, w, 0.25, 4, 3, qs, qg, kg)
    vis = O.visibility(2, 64, 16, 4, qs, qg, kg)
    assert np.all(sc[vis] == 0.0) and np.all(sc[~vis] == -np.inf)
    for b in range(2):
        for s in range(64):
            v = np.nonzero(vis[b, s])[0][:3].tolist()
            assert idx[b, s].tolist() == v + [-1] * (3 - len(v))


def test_linear_in_weights():
    q, k, w, qs, qg, kg = _prob(3)
    w2 = np.random.default_rng(9).standard_normal(w.shape)
    a = O.index_scores(q, k, w, 0.25, 4, qs, qg, kg)
    b = O.index_scores(q, k, w2, 0.25, 4, qs, qg, kg)
    c = O.index_scores(q, k, 2.0 * w - 3.0 * w2, 0.25, 4, qs, qg, kg)
    fin = np.isfinite(a)
    np.testing.assert_allclose(c[fin], 2.0 * a[fin] - 3.0 * b[fin], rtol=1e-12, atol=1e-12)


def test_head_permutation_invariance():
    q, k, w, qs, qg, kg = _prob(4, H=6)
    perm = np.array([3, 0, 5, 1, 4, 2])
    a = O.index_scores(q, k, w, 0.25, 4, qs, qg, kg)
    b = O.index_scores(q[:, perm], k, w[:, :, perm], 0.25, 4, qs, qg, kg)
    fin = np.isfinite(a)
    np.testing.assert_allclose(a[fin], b[fin], rtol=1e-12, atol=1e-12)
    # a mismatched permutation (q permuted, w not) must change the scores
    c = O.index_scores(q[:, perm], k, w, 0.25, 4, qs, qg, kg)
    assert not np.allclose(a[fin], c[fin])


def test_head_split_additivity():
    q, k, w, qs, qg, kg = _prob(5, segs=False, H=8)
    full = O.index_scores(q, k, w, 0.25, 4, qs)
    lo = O.index_scores(q[:, :4], k, w[:, :, :4], 0.25, 4, qs)
    hi = O.index_scores(q[:, 4:], k, w[:, :, 4:], 0.25, 4, qs)
    fin = np.isfinite(full)
    np.testing.assert_allclose(full[fin], lo[fin] + hi[fin], rtol=1e-12, atol=1e-12)


def test_scale_homogeneity_and_relu_placement():
    q, k, w, qs, qg, kg = _prob(6, segs=False)
    a = O.index_scores(q, k, w, 0.25, 4, qs)
    b = O.index_scores(q, k, w, 0.5, 4, qs)
    fin = np.isfinite(a)
    np.testing.assert_allclose(b[fin], 2.0 * a[fin], rtol=1e-12, atol=1e-12)
    # ReLU acts per head before the weighted sum: negating q flips which
    # logits survive, so the scores are not simply negated
    c = O.index_scores(-q, k, w, 0.25, 4, qs)
    assert not np.allclose(c[fin], -a[fin])


def test_packed_equals_unpacked_documents():
    rng = np.random.default_rng(11)
    r, S, H, D = 4, 96, 3, 8
    W = S // r
    cuts = [0, 24, 56, 96]  # document boundaries, multiples of r
    q = rng.standard_normal((1, H, S, D))
    k = rng.standard_normal((1, W, D))
    w = rng.standard_normal((1, S, H))
    q_seg = np.zeros((1, S), dtype=np.int32)
    for i, c in enumerate(cuts[1:-1]):
        q_seg[0, c:] = i + 1
    kv_seg = q_seg[:, np.arange(W) * r + r - 1]
    top_k = 5
    sc, idx = O.index_topk(q, k, w, 0.3, r, top_k, None, q_seg, kv_seg)
    for a, b in zip(cuts[:-1], cuts[1:]):
        e0, e1 = a // r, b // r
        sd, idd = O.index_topk(q[:, :, a:b], k[:, e0:e1], w[:, a:b], 0.3, r, top_k)
        np.testing.assert_array_equal(sc[0, a:b, e0:e1], sd[0])
        assert np.all(sc[0, a:b, :e0] == -np.inf) and np.all(sc[0, a:b, e1:] == -np.inf)
        shifted = np.where(idd[0] >= 0, idd[0] + e0, -1)
        np.testing.assert_array_equal(idx[0, a:b], shifted)


def test_row_slice_equals_full_run():
    q, k, w, _, qg, kg = _prob(8, segs=True)
    full_sc, full_idx = O.index_topk(q, k, w, 0.25, 4, 6, None, qg, kg)
    s0, s1 = 17, 45
    start = np.array([s0, s0])
    sc, idx = O.index_topk(q[:, :, s0:s1], k, w[:, s0:s1], 0.25, 4, 6, start, qg[:, s0:s1], kg)
    np.testing.assert_array_equal(sc, full_sc[:, s0:s1])
    np.testing.assert_array_equal(idx, full_idx[:, s0:s1])
    rows = np.arange(s0, s1)
    sc2 = O.index_scores(q, k, w, 0.25, 4, None, qg, kg, rows=rows)
    np.testing.assert_array_equal(sc2, full_sc[:, s0:s1])


def test_rows_with_few_visible_return_visible_set():
    q, k, w, qs, qg, kg = _prob(9)
    top_k = 6
    sc, idx = O.index_topk(q, k, w, 0.25, 4, top_k, qs, qg, kg)
    vis = O.visibility(2, 64, 16, 4, qs, qg, kg)
    for b in range(2):
        for s in range(64):
            v = np.nonzero(vis[b, s])[0].tolist()
            if len(v) <= top_k:
                assert idx[b, s].tolist() == v + [-1] * (top_k - len(v))


def test_decode_start_makes_all_visible():
    vis = O.visibility(2, 1, 32768, 4, q_start=np.array([131071, 131071]))
    assert vis.all()
    vis = O.visibility(1, 1, 32768, 4, q_start=np.array([131070]))
    assert vis[0, 0, :32767].all() and not vis[0, 0, 32767]


def test_gather_selected_matches_loops():
    rng = np.random.default_rng(12)
    k = rng.standard_normal((2, 9, 5))
    idx = rng.integers(-1, 9, size=(2, 4, 3))
    out = O.gather_selected(k, idx)
    for b in range(2):
        for s in range(4):
            for i in range(3):
                t = idx[b, s, i]
                expect = np.zeros(5) if t < 0 else k[b, t]
                assert np.array_equal(out[b, s, i], expect)


# --------------------------------------------------------------------------- backward
def test_backward_hand_example():
    g, q, k, w, _ = _hand()
    ex = g["backward_example"]
    G = np.zeros((1, g["S"], g["W"]))
    for s_, t_, v in ex["g_entries"]:
        G[0, s_, t_] = v
    dq, dk, dw = O.index_scores_vjp(q, k, w, g["scale"], g["compress_rate"], G)
    edq, edk, edw = np.zeros_like(dq), np.zeros_like(dk), np.zeros_like(dw)
    for h, s_, d, v in ex["expected_dq_nonzero"]:
        edq[0, h, s_, d] = v
    for t_, d, v in ex["expected_dk_nonzero"]:
        edk[0, t_, d] = v
    for s_, h, v in ex["expected_dw_nonzero"]:
        edw[0, s_, h] = v
    assert np.array_equal(dq, edq) and np.array_equal(dk, edk) and np.array_equal(dw, edw)


def _loss(q, k, w, scale, r, G, q_start=None, q_seg=None, kv_seg=None):
    sc = O.index_scores(q, k, w, scale, r, q_start, q_seg, kv_seg)
    return float(np.where(np.isfinite(sc), G * np.where(np.isfinite(sc), sc, 0.0), 0.0).sum())


@pytest.mark.parametrize("seed", range(3))
def test_backward_finite_differences(seed):
    rng = np.random.default_rng(300 + seed)
    B, H, S, D, W, r = 1, 2, 6, 3, 4, 2
    segs = seed == 1
    start = [3] if seed == 2 else None
    q, k, w, q_start, q_seg, kv_seg = _rand_problem(rng, B, H, S, D, W, r, segs, start)
    G = rng.standard_normal((B, S, W))
    scale = 0.61
    c = O.scale_value(scale)
    x = np.einsum("bhsd,btd->bhst", q, k)
    assert np.min(np.abs(c * x)) > 1e-3  # away from the ReLU kink
    dq, dk, dw = O.index_scores_vjp(q, k, w, scale, r, G, q_start, q_seg, kv_seg)
    eps = 1e-6
    for arr, grad in ((q, dq), (k, dk), (w, dw)):
        for i in np.ndindex(arr.shape):
            old = arr[i]
            arr[i] = old + eps
            lp = _loss(q, k, w, scale, r, G, q_start, q_seg, kv_seg)
            arr[i] = old - eps
            lm = _loss(q, k, w, scale, r, G, q_start, q_seg, kv_seg)
            arr[i] = old
            assert abs((lp - lm) / (2 * eps) - grad[i]) < 1e-6 * (1 + abs(grad[i])), (i, grad[i])


@pytest.mark.parametrize("seed", range(3))
def test_backward_euler_homogeneity(seed):
    # score is positively homogeneous of degree 1 in q, in k and in w, so
    # sum(q*dq) = sum(k*dk) = sum(w*dw) = sum(g*score) over visible entries
    rng = np.random.default_rng(400 + seed)
    q, k, w, q_start, q_seg, kv_seg = _rand_problem(rng, 2, 3, 20, 8, 9, 2, seed == 1, [5, 0] if seed == 2 else None)
    G = rng.standard_normal((2, 20, 9))
    dq, dk, dw = O.index_scores_vjp(q, k, w, 0.3, 2, G, q_start, q_seg, kv_seg)
    L = _loss(q, k, w, 0.3, 2, G, q_start, q_seg, kv_seg)
    for a, d in ((q, dq), (k, dk), (w, dw)):
        assert abs(float((a * d).sum()) - L) < 1e-10 * (1 + abs(L))


def test_backward_linear_in_g_and_blind_to_masked_g():
    rng = np.random.default_rng(7)
    q, k, w, q_start, q_seg, kv_seg = _rand_problem(rng, 1, 2, 16, 4, 8, 2, True, None)
    G1, G2 = rng.standard_normal((2, 1, 16, 8))
    a = O.index_scores_vjp(q, k, w, 0.5, 2, G1 + 2.0 * G2, q_start, q_seg, kv_seg)
    b1 = O.index_scores_vjp(q, k, w, 0.5, 2, G1, q_start, q_seg, kv_seg)
    b2 = O.index_scores_vjp(q, k, w, 0.5, 2, G2, q_start, q_seg, kv_seg)
    for x, y, z in zip(a, b1, b2):
        np.testing.assert_allclose(x, y + 2.0 * z, rtol=1e-12, atol=1e-12)
    vis = O.visibility(1, 16, 8, 2, q_start, q_seg, kv_seg)
    G3 = np.where(vis, G1, 1e6)  # anything at masked entries
    c = O.index_scores_vjp(q, k, w, 0.5, 2, G3, q_start, q_seg, kv_seg)
    for x, y in zip(c, b1):
        assert np.array_equal(x, y)

"""CPU oracle for the CSA indexer score + top-k path (test infrastructure).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
link this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It
shares no code with the CUDA library and never reads a value produced there
except where a test hands it the GPU's own scores to re-run the selector.

What it computes (float64 throughout, from the exact stored bf16/fp32 input
values):

* ``index_scores`` -- the head-reduced indexer score of "Add StreamIndex Kernel
  for CSA [Deepseek v4]" (Description: the fused per-head q.k^T, activation,
  weighting by ``weights[b,s,h]`` and sum over heads; the kernel's output block
  is ``(block_q, block_w)`` of a ``[B,S,W]`` tensor, BlockSpec review hunk)::

      score[b,s,t] = sum_h w[b,s,h] * ReLU(scale * <q[b,h,s,:], k[b,t,:]>)

  The pages never name the activation; ReLU is the reading taken here.
* ``visibility`` -- the future mask of "DSV4: Add indexer_save_selection and
  indexer_sharded_topk" (review hunk: ``entry >= causal_threshold`` is masked)
  with ``causal_threshold = (pos + 1) // compress_rate`` (reading: compressed
  entry t covers tokens ``t*r .. t*r+r-1`` and becomes visible once its last
  token is at or before the query position), plus the packed-document segment
  mask of the same hunk (entries of another document are masked).
* ``select_topk`` -- per query row, the ``top_k`` best visible entries
  (same page, Description: the selection handed to sparse attention).
  Readings: larger score first, ties to the lower entry index, comparison by
  value (``-0.0 == +0.0``), output sorted ascending by entry index and padded
  with ``-1`` when fewer than ``top_k`` entries are visible.  It is a full
  stable sort, not a selection algorithm.
* ``brute_force_scores`` -- the same definition written as plain Python loops
  over (b, s, t, h, d), for tiny shapes only.
* ``index_scores_vjp`` -- the backward of the score step: for a cotangent
  ``g[B,S,W]`` of the scores, the gradients ``dq, dk, dw`` of
  ``sum(g * score)`` over the visible entries ("Add StreamIndex Kernel for CSA
  [Deepseek v4]", Description: the custom_vjp whose backward is the
  autodiff of the reference computation).  Readings: masked entries are
  constants (``-inf``) and take no gradient, so ``g`` is used only where
  visible; the ReLU derivative at 0 is 0.

Parity pins (see ``tests/test_oracle.py``): for the backward, central finite
differences on tiny shapes, Euler's identity for the degree-1 positive
homogeneity of the score in q, in k and in w separately (each of
``sum(q*dq)``, ``sum(k*dk)``, ``sum(w*dw)`` equals ``sum(g*score)``),
linearity in g and independence of g at masked entries.  For the forward: a hand-worked 2-head / 4-entry
example, brute force on tiny shapes, the H=1 / w=1 / scale=1 special case
reducing to ``max(Q K^T, 0)`` and ``argsort``, and invariants (masked entries
never selected, w=0 gives zero scores and the lowest visible indices,
linearity in w, head permutation, head-split additivity, zero padding of D/H,
homogeneity in scale, packed == unpacked documents, row slice == full run).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np


def _f64(x):
    return None if x is None else np.asarray(x, dtype=np.float64)


def scale_value(scale: float) -> float:
    """The scale as the library receives it: rounded to float32, then widened."""
    return float(np.float64(np.float32(scale)))


def causal_threshold(pos: np.ndarray, compress_rate: int) -> np.ndarray:
    """Number of compressed entries visible at absolute position ``pos``.

    Entry t holds tokens ``t*r .. t*r+r-1``; it is visible once token
    ``t*r+r-1 <= pos``, i.e. ``t < (pos+1)//r`` (the ``causal_threshold`` of
    the future-mask hunk on "DSV4: Add indexer_save_selection and
    indexer_sharded_topk"; formula: the reading stated in the module doc).
    """
    return (np.asarray(pos, dtype=np.int64) + 1) // int(compress_rate)


def visibility(B: int, S: int, W: int, compress_rate: int,
               q_start: Optional[np.ndarray] = None,
               q_seg: Optional[np.ndarray] = None,
               kv_seg: Optional[np.ndarray] = None,
               rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """Boolean ``[B, R, W]`` visibility (``R = len(rows)`` or ``S``).

    ``vis[b,s,t] = t < (q_start[b]+s+1)//r  and  (no segments or
    q_seg[b,s] == kv_seg[b,t])`` -- future mask and segment mask of the mask
    review hunk on "DSV4: Add indexer_save_selection and indexer_sharded_topk".
    """
    rows = np.arange(S) if rows is None else np.asarray(rows, dtype=np.int64)
    start = np.zeros(B, dtype=np.int64) if q_start is None else np.asarray(q_start, dtype=np.int64)
    pos = start[:, None] + rows[None, :]                       # [B, R]
    thr = causal_threshold(pos, compress_rate)                  # [B, R]
    t = np.arange(W, dtype=np.int64)
    vis = t[None, None, :] < thr[:, :, None]                    # entry >= threshold is masked
    if q_seg is not None:
        qs = np.asarray(q_seg)[:, rows]                         # [B, R]
        ks = np.asarray(kv_seg)                                 # [B, W]
        vis &= qs[:, :, None] == ks[:, None, :]
    return vis


def index_scores(q, k, w, scale: float, compress_rate: int,
                 q_start=None, q_seg=None, kv_seg=None,
                 rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """float64 ``[B, R, W]`` head-reduced scores, ``-inf`` where masked.

    ``q [B,H,S,D]``, ``k [B,W,D]``, ``w [B,S,H]`` hold the exact input values.
    For each batch and head one ``[R,D] x [D,W]`` product (a library matmul is
    the contraction step), then ``ReLU(scale * x)`` weighted by ``w[b,s,h]``
    and summed over heads; masked entries are then set to ``-inf``.
    """
    Q, K, Wt = _f64(q), _f64(k), _f64(w)
    B, H, S, D = Q.shape
    W = K.shape[1]
    rows = np.arange(S) if rows is None else np.asarray(rows, dtype=np.int64)
    c = scale_value(scale)
    out = np.zeros((B, len(rows), W), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            x = Q[b, h][rows] @ K[b].T                          # [R, W] per-head logits
            out[b] += Wt[b, rows, h][:, None] * np.maximum(c * x, 0.0)
    vis = visibility(B, S, W, compress_rate, q_start, q_seg, kv_seg, rows)
    out[~vis] = -np.inf
    return out


def select_topk(scores, top_k: int) -> np.ndarray:
    """int64 ``[..., top_k]`` selection from ``[..., W]`` scores.

    Visible means ``score > -inf``.  Entries are ordered by a stable sort on
    ``-score`` (so equal values keep ascending entry order: ties go to the
    lower index, and ``-0.0`` equals ``+0.0`` because the sort compares
    values).  The first ``min(top_k, visible)`` are kept, sorted ascending by
    index, and the row is padded with ``-1``.
    """
    sc = _f64(scores)
    lead = sc.shape[:-1]
    W = sc.shape[-1]
    flat = sc.reshape(-1, W)
    vis = flat > -np.inf
    nvis = vis.sum(axis=1)
    key = np.where(vis, -flat, np.inf)                          # invisible sorts last
    order = np.argsort(key, axis=1, kind="stable")
    out = np.full((flat.shape[0], top_k), -1, dtype=np.int64)
    take = min(top_k, W)
    big = np.iinfo(np.int64).max
    chosen = order[:, :take].astype(np.int64)
    keep = np.arange(take)[None, :] < nvis[:, None]
    chosen = np.sort(np.where(keep, chosen, big), axis=1)
    chosen[chosen == big] = -1
    out[:, :take] = chosen
    return out.reshape(*lead, top_k)


def index_topk(q, k, w, scale, compress_rate, top_k, q_start=None, q_seg=None,
               kv_seg=None, rows=None):
    """Scores then selection: the whole hot path for the given rows."""
    sc = index_scores(q, k, w, scale, compress_rate, q_start, q_seg, kv_seg, rows)
    return sc, select_topk(sc, top_k)


def gather_selected(k, idx) -> np.ndarray:
    """``out[b,s,i,:] = k[b, idx[b,s,i], :]``, zeros where ``idx == -1``: the
    selected compressed rows handed to sparse attention ("DSV4: Add
    indexer_save_selection and indexer_sharded_topk", Description)."""
    K = np.asarray(k)
    I = np.asarray(idx)
    B, W, D = K.shape
    out = np.zeros(I.shape + (D,), dtype=K.dtype)
    for b in range(B):
        sel = I[b] >= 0
        out[b][sel] = K[b][I[b][sel]]
    return out


def visible_counts(B, S, W, compress_rate, q_start=None, q_seg=None, kv_seg=None, rows=None):
    """``v[b,s]``: number of visible entries of each row."""
    return visibility(B, S, W, compress_rate, q_start, q_seg, kv_seg, rows).sum(axis=-1)


def brute_force_scores(q, k, w, scale, compress_rate, q_start=None, q_seg=None, kv_seg=None):
    """The score definition as plain nested loops (tiny shapes only)."""
    Q, K, Wt = _f64(q), _f64(k), _f64(w)
    B, H, S, D = Q.shape
    W = K.shape[1]
    c = scale_value(scale)
    out = [[[0.0] * W for _ in range(S)] for _ in range(B)]
    for b in range(B):
        start = 0 if q_start is None else int(q_start[b])
        for s in range(S):
            for t in range(W):
                if t * compress_rate + compress_rate - 1 > start + s:
                    out[b][s][t] = -np.inf
                    continue
                if q_seg is not None and int(q_seg[b][s]) != int(kv_seg[b][t]):
                    out[b][s][t] = -np.inf
                    continue
                acc = 0.0
                for h in range(H):
                    dot = 0.0
                    for d in range(D):
                        dot += float(Q[b, h, s, d]) * float(K[b, t, d])
                    x = c * dot
                    acc += float(Wt[b, s, h]) * (x if x > 0.0 else 0.0)
                out[b][s][t] = acc
    return np.array(out, dtype=np.float64)


def index_scores_vjp(q, k, w, scale: float, compress_rate: int, g,
                     q_start=None, q_seg=None, kv_seg=None):
    """float64 ``(dq [B,H,S,D], dk [B,W,D], dw [B,S,H])`` for the cotangent
    ``g [B,S,W]`` of the visible scores.

    With ``x = q[b,h,s,:] . k[b,t,:]`` and ``gm = g`` on visible entries, 0
    elsewhere (chain rule through ``score = sum_h w * ReLU(scale * x)``):

        dw[b,s,h] = sum_t gm[b,s,t] * ReLU(scale * x)
        dx        = gm[b,s,t] * w[b,s,h] * scale * [scale * x > 0]
        dq[b,h]   = dx @ k[b]          dk[b] = sum_h dx^T @ q[b,h]

    one library matmul per contraction, per batch and head.
    """
    Q, K, Wt, G = _f64(q), _f64(k), _f64(w), _f64(g)
    B, H, S, D = Q.shape
    W = K.shape[1]
    c = scale_value(scale)
    vis = visibility(B, S, W, compress_rate, q_start, q_seg, kv_seg)
    gm = np.where(vis, G, 0.0)
    dq = np.zeros_like(Q)
    dk = np.zeros_like(K)
    dw = np.zeros((B, S, H), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            x = Q[b, h] @ K[b].T                                # [S, W]
            cx = c * x
            dw[b, :, h] = (gm[b] * np.maximum(cx, 0.0)).sum(axis=1)
            dx = gm[b] * Wt[b, :, h][:, None] * c * (cx > 0.0)
            dq[b, h] = dx @ K[b]
            dk[b] += dx.T @ Q[b, h]
    return dq, dk, dw

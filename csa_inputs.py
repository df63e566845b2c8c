"""Seeded synthetic inputs for the CSA indexer workloads.

This module only draws random numbers and lays them out; it holds none of the
indexer's arithmetic.  Both the CUDA path (tests, ``bench.py``) and the CPU
oracle consume what it returns, so the two always see identical input bits.

Recipe (one ``torch.Generator('cpu')`` seeded per problem, drawn in this order):
  1. ``q = randn(B, H, S, D)``       -> bf16 (round to nearest even)
  2. ``k = randn(B, W, D)``          -> bf16
  3. ``w = randn(B, S, H) * sigma_w`` -> ``w_dtype`` (bf16 or fp32)
  4. packed-document segment ids (only when ``docs`` is given): per batch row,
     ``n = randint(docs[0], docs[1] + 1)`` documents, ``n - 1`` distinct cut
     points drawn uniformly from the multiples of ``compress_rate`` in
     ``(0, S)``; ``q_seg[s]`` is the document index of token ``s`` and
     ``kv_seg[t]`` is the document of the last token of compressed block ``t``
     (token ``t * r + r - 1``).

The workloads follow the shapes of the DeepSeek-V4 CSA indexer described on
"Add StreamIndex Kernel for CSA [Deepseek v4]" (q head-major ``[B,H,S,D]``,
compressed ``[B,W,D]``, weights ``[B,S,H]``, Description and BlockSpec review
hunk) and "DSV4: Add indexer_save_selection and indexer_sharded_topk"
(sequence length 16384, packed documents, autoregressive decode).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Tuple

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic indexer problem (shapes, dtypes and draw parameters)."""

    name: str
    B: int
    S: int
    W: int
    H: int
    D: int
    compress_rate: int
    top_k: int
    w_dtype: str  # "bf16" | "f32"
    sigma_w: float
    scale: float
    q_start: Optional[int] = None  # same start position for every batch row; None = 0
    docs: Optional[Tuple[int, int]] = None  # (min, max) documents per row
    seed: int = 0

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _cfg(name, B, S, r, H, D, top_k, w_dtype, sigma_w, W=None, q_start=None, docs=None):
    return Workload(name=name, B=B, S=S, W=(S // r) if W is None else W, H=H, D=D,
                    compress_rate=r, top_k=top_k, w_dtype=w_dtype, sigma_w=sigma_w,
                    scale=1.0 / math.sqrt(D), q_start=q_start, docs=docs)


# The five workloads: a tiny parity case, a mid-size prefill, the long-context
# prefill (sequence 16384), packed documents and single-row decode; then two
# longer prefills (sequences 32768 and 65536).
WORKLOADS = {
    "tiny": _cfg("tiny", 1, 256, 4, 4, 32, 16, "f32", 0.5),
    "prefill_4k": _cfg("prefill_4k", 1, 4096, 4, 64, 128, 512, "bf16", 1.0 / 8),
    "prefill_16k": _cfg("prefill_16k", 2, 16384, 4, 64, 128, 2048, "bf16", 1.0 / 8),
    "packed_8k": _cfg("packed_8k", 4, 8192, 4, 64, 128, 1024, "bf16", 1.0 / 8, docs=(3, 8)),
    "decode_32k": _cfg("decode_32k", 64, 1, 4, 64, 128, 2048, "bf16", 1.0 / 8,
                       W=32768, q_start=131071),
    # longer prefills (rows of up to 8192 / 16384 compressed entries), the
    # same distributions: the fused kernel's long-row mode
    "prefill_32k": _cfg("prefill_32k", 1, 32768, 4, 64, 128, 2048, "bf16", 1.0 / 8),
    "prefill_64k": _cfg("prefill_64k", 1, 65536, 4, 64, 128, 2048, "bf16", 1.0 / 8),
}


@dataclasses.dataclass
class Inputs:
    """CPU tensors of one problem.  q, k are bf16; w is bf16 or fp32."""

    wl: Workload
    q: torch.Tensor            # [B, H, S, D] bf16
    k: torch.Tensor            # [B, W, D] bf16
    w: torch.Tensor            # [B, S, H] bf16 | fp32
    q_seg: Optional[torch.Tensor]   # [B, S] int32
    kv_seg: Optional[torch.Tensor]  # [B, W] int32
    q_start: Optional[torch.Tensor]  # [B] int64


def _segments(gen: torch.Generator, wl: Workload):
    B, S, W, r = wl.B, wl.S, wl.W, wl.compress_rate
    lo, hi = wl.docs
    q_seg = torch.empty(B, S, dtype=torch.int32)
    kv_seg = torch.empty(B, W, dtype=torch.int32)
    n_slots = S // r - 1  # multiples of r strictly inside (0, S)
    for b in range(B):
        n = int(torch.randint(lo, hi + 1, (1,), generator=gen))
        n = max(1, min(n, n_slots + 1))
        cuts = torch.randperm(n_slots, generator=gen)[: n - 1] + 1
        cuts = torch.sort(cuts * r).values
        doc = torch.zeros(S, dtype=torch.int32)
        for c in cuts.tolist():
            doc[c:] += 1
        q_seg[b] = doc
        last_tok = torch.arange(W, dtype=torch.int64) * r + (r - 1)
        kv_seg[b] = doc[last_tok.clamp(max=S - 1)]
    return q_seg, kv_seg


def make_inputs(wl: Workload) -> Inputs:
    """Draw the problem's inputs on the CPU, in the recipe's order."""
    gen = torch.Generator("cpu").manual_seed(wl.seed)
    q = torch.randn(wl.B, wl.H, wl.S, wl.D, generator=gen).to(torch.bfloat16)
    k = torch.randn(wl.B, wl.W, wl.D, generator=gen).to(torch.bfloat16)
    w = torch.randn(wl.B, wl.S, wl.H, generator=gen) * wl.sigma_w
    w = w.to(torch.bfloat16 if wl.w_dtype == "bf16" else torch.float32)
    q_seg = kv_seg = None
    if wl.docs is not None:
        q_seg, kv_seg = _segments(gen, wl)
    q_start = None
    if wl.q_start is not None:
        q_start = torch.full((wl.B,), wl.q_start, dtype=torch.int64)
    return Inputs(wl, q, k, w, q_seg, kv_seg, q_start)


def to_f64(t: torch.Tensor):
    """Exact numpy float64 copy of a bf16/fp32 tensor (no rounding)."""
    return t.to(torch.float64).numpy()

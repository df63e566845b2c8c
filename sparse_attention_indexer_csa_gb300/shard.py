"""Partition of one indexer problem's query rows across ranks.

Query rows are independent: a rank that owns rows [s0, s1) of every sequence
passes q and w of those rows with q_start = s0 (added to the sequences' own
start) and gets exactly those rows' selections -- the row-sharded top-k of
"DSV4: Add indexer_save_selection and indexer_sharded_topk" (Description:
query rows are sharded for the masking and the top-k, and the selection is
unchanged).  No data moves between ranks to compute a shard; gathering the
shards' indices afterwards is the caller's choice.

Later rows see more compressed entries, so equal row counts are unequal
work.  The cut points split the rows' visible-entry counts (the future
mask's count, the work of the score step) evenly and fall on multiples of
four rows, the row block of the kernels.
"""
from __future__ import annotations

from typing import List, Tuple


def visible_entries(s: int, W: int, compress_rate: int, q_start: int = 0) -> int:
    """Entries row s can see under the future mask (segments not counted)."""
    v = (q_start + s + 1) // compress_rate
    return max(0, min(W, v))


def row_shards(S: int, W: int, compress_rate: int, n: int, q_start: int = 0,
               block: int = 4) -> List[Tuple[int, int]]:
    """`n` contiguous row ranges [s0, s1) covering 0..S, balanced by visible
    entries, with inner cut points on multiples of `block`.  Ranges may be
    empty when S is small."""
    if n < 1:
        raise ValueError("n must be >= 1")
    cum = [0]
    for s in range(S):
        cum.append(cum[-1] + visible_entries(s, W, compress_rate, q_start))
    total = cum[-1]
    cuts = [0]
    s = 0
    for r in range(1, n):
        target = total * r / n
        while s < S and cum[s] < target:
            s += 1
        c = min(S, max(cuts[-1], (s // block) * block))
        cuts.append(c)
    cuts.append(S)
    return [(cuts[i], cuts[i + 1]) for i in range(n)]

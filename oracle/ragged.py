"""Row layout of one selectively batched iteration and its work counts.

Selective batching flattens the new tokens of all requests into one
[sum L_i, H] tensor instead of a padded [B, L, H] one (Orca walk-through,
Figure 5: four requests, seven rows).  Row order is the batch order; the
rows of request i are row_off[i] .. row_off[i+1]-1, and row j of request i
sits at position c_i + j of its sequence.  Attention of that row reads the
request's keys 0 .. c_i + j (causal, itself included).

Work counts follow CS349D Lecture 2, section 3.2 and Exercise 4: useful
(query, key) pairs per head are c_i + 1 for a decode row and L(L+1)/2 for a
prefill of L tokens; a padded layout pads every request to max L_i queries
and max (c_i + L_i) keys.
"""
from typing import Dict, List, Sequence, Tuple


def layout(batch: Sequence[Tuple[int, int]]) -> Dict[str, List[int]]:
    """batch = [(L_i, c_i)] in batch order -> row offsets, per-row request
    index and position, each request's last row."""
    row_off = [0]
    row_req: List[int] = []
    row_pos: List[int] = []
    for i, (L, c) in enumerate(batch):
        row_off.append(row_off[-1] + L)
        row_req += [i] * L
        row_pos += [c + j for j in range(L)]
    last_row = [row_off[i + 1] - 1 for i in range(len(batch))]
    return {"row_off": row_off, "row_req": row_req, "row_pos": row_pos, "last_row": last_row,
            "n_rows": row_off[-1]}


def useful_pairs(batch: Sequence[Tuple[int, int]]) -> int:
    """Causal (query, key) pairs per head: sum over rows of (position + 1)."""
    return sum(c + j + 1 for (L, c) in batch for j in range(L))


def padded_rows(batch: Sequence[Tuple[int, int]]) -> int:
    return len(batch) * max(L for L, _ in batch)


def padded_pairs(batch: Sequence[Tuple[int, int]]) -> int:
    return len(batch) * max(L for L, _ in batch) * max(L + c for L, c in batch)

"""Dispatch of token slots to per-expert contiguous rows, by definition.

Test infrastructure only (see oracle/__init__.py).

On the pages, dispatch is the all-to-all that carries each token's
activations to the GPU holding its expert (Moreh report, sections
"Overview" and "Compute-communication overlap").  On one GPU it becomes a
permutation into per-expert contiguous rows.  The layout read here:
  * slots: routed slot i = t*k + j for token t and choice j; the shared
    expert s of token t is slot T*k + s*T + t;
  * rows: routed rows are the routed slots stably sorted by expert id, so
    within an expert the rows are in increasing slot order; shared expert s
    occupies the T rows after every routed row and earlier shared expert;
  * expert_offsets[g] is the first row of group g (routed experts first,
    then the shared experts), expert_offsets[G] = total rows;
  * src_of_row[r] is the slot of row r, row_of_slot[t, j] the row of slot
    (t, j).
"""
from __future__ import annotations

import numpy as np


def permute(topk_ids: np.ndarray, num_experts: int, num_shared: int):
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, k = ids.shape
    R = T * k
    flat = ids.reshape(-1)
    counts = np.bincount(flat, minlength=num_experts)[:num_experts]
    group_rows = np.concatenate([counts, np.full(num_shared, T)]).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(group_rows)]).astype(np.int32)
    order = np.argsort(flat, kind="stable")           # rows -> routed slots
    src_of_row = np.concatenate([order, R + np.arange(num_shared * T)]).astype(np.int32)
    row_of_slot = np.empty(R, dtype=np.int32)
    row_of_slot[order] = np.arange(R, dtype=np.int32)
    return offsets, src_of_row, row_of_slot.reshape(T, k)


def token_of_slot(slot: np.ndarray, T: int, k: int) -> np.ndarray:
    slot = np.asarray(slot, dtype=np.int64)
    return np.where(slot < T * k, slot // k, (slot - T * k) % T)

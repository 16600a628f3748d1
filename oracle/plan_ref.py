"""Plain restatement of the occupancy-pinned split-KV plan.

TEST INFRASTRUCTURE ONLY: imported by tests/, the smoke check and the
benchmark's CPU legs, never by the library.  It shares no code with the C++
plan inside the CUDA library; the two are compared field by field.

Source: the "mjolnir/t5_decode.py" page, `plan_split_kv` and `SplitPlan`
(host helpers section).  What the rule asks for, as its documentation
states it:

* KV is cut into tiles of 128 rows; a sequence owns ``max(1, ceil(L / 128))``
  tiles (an empty sequence still owns one, so its output rows are written).
* The grid is (work items, q tiles, kv heads); one wave of it holds
  ``slots = max(1, sm_count * ctas_per_sm // (h_k * n_q_tiles))`` items.
* Every sequence is cut into consecutive chunks of the same size (the last
  one may be shorter).  The chunk is never smaller than ``min_chunk_tiles``
  nor than ``ceil(T / max_splits)`` (T: the longest sequence's tiles), so no
  sequence has more than max_splits chunks.
* A forced split count cuts the longest sequence into that many chunks (still
  above the floor).  Otherwise nothing is split when max_splits is 1 or when
  the batch already has at least one item per slot; else the chunk is the
  smallest size (above the floor) whose total number of chunks fits in one
  wave.
* Work items are ordered longest first; among equal lengths, sequence
  ascending, then chunk index ascending.  Optional padding appends empty
  (0, 0, 0, 0) items.

This module writes those statements as directly as possible: the chunk is
found by trying every candidate size upward from the floor, and the order is
an explicit three-part sort key.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Sequence, Tuple

TILE_ROWS = 128


@dataclass
class PlanRef:
    work: List[Tuple[int, int, int, int]] = field(default_factory=list)
    n_splits: List[int] = field(default_factory=list)
    chunk_tiles: int = 0
    slots: int = 0


def _tiles(length: int) -> int:
    """128-row tiles of a sequence of `length` keys (at least one)."""
    whole, rest = divmod(int(length), TILE_ROWS)
    return max(1, whole + (1 if rest else 0))


def _pieces(tiles: int, chunk: int) -> int:
    """Chunks of `chunk` tiles that cover `tiles` tiles."""
    n = 0
    covered = 0
    while covered < tiles:
        covered += chunk
        n += 1
    return n


def plan_ref(
    seq_lens: Sequence[int],
    h_k: int,
    n_q_tiles: int,
    sm_count: int,
    ctas_per_sm: int = 1,
    max_splits: int = 16,
    force_splits: int = 0,
    min_chunk_tiles: int = 1,
    pad_to: int = 0,
) -> PlanRef:
    tiles = [_tiles(L) for L in seq_lens]
    longest = max(tiles)
    slots = max(1, (sm_count * ctas_per_sm) // (h_k * n_q_tiles))
    # the floor: at most max_splits chunks for the longest sequence
    floor_chunk = min_chunk_tiles
    while _pieces(longest, floor_chunk) > max_splits:
        floor_chunk += 1

    if force_splits > 0:
        chunk = floor_chunk
        while _pieces(longest, chunk) > force_splits:
            chunk += 1
    elif max_splits == 1 or len(tiles) >= slots:
        chunk = longest
    else:
        # every candidate from the floor upward; `longest` always fits (one
        # chunk per sequence, fewer sequences than slots here)
        chunk = floor_chunk
        while chunk < longest and sum(_pieces(t, chunk) for t in tiles) > slots:
            chunk += 1

    items = []
    n_splits = []
    for b, t in enumerate(tiles):
        begin, k = 0, 0
        while begin < t:
            end = min(t, begin + chunk)
            items.append((b, begin, end, k))
            begin, k = end, k + 1
        n_splits.append(k)
    items.sort(key=lambda it: (-(it[2] - it[1]), it[0], it[3]))
    if pad_to:
        if pad_to < len(items):
            raise ValueError(f"pad_to {pad_to} < {len(items)} work items")
        items = items + [(0, 0, 0, 0)] * (pad_to - len(items))
    if max(n_splits) > max_splits:
        raise ValueError("plan exceeds max_splits")
    return PlanRef(items, n_splits, chunk, slots)

"""Plain restatement of the occupancy-pinned split-KV plan.

TEST INFRASTRUCTURE ONLY: imported by tests/, the smoke check and the
benchmark's CPU legs, never by the library.  It shares no code with the C++
plan inside the CUDA library; the two are compared field by field.

Source: the "mjolnir/t5_decode.py" page, `plan_split_kv` and `SplitPlan`
(host helpers section).  The steps, in the page's order:

1. Every sequence has ``max(1, ceil(L / 128))`` KV tiles of 128 rows (a
   sequence of length 0 still owns one tile, so its rows get written).
2. One wave of the grid ``(work items, q tiles, kv heads)`` holds
   ``slots = max(1, sm_count * ctas_per_sm // (h_k * n_q_tiles))`` items.
3. The chunk size (tiles per work item) is at least
   ``lo = max(min_chunk_tiles, ceil(T / max_splits))`` with T the longest
   sequence's tile count, so no sequence is cut into more than max_splits.
4. ``force_splits > 0`` takes ``max(lo, ceil(T / force_splits))``; a batch
   that already fills the wave, or max_splits == 1, takes ``T`` (no split);
   otherwise the chunk is the smallest value >= lo whose chunk total
   ``sum(ceil(t / chunk))`` fits in ``slots`` (T always fits: one per
   sequence, fewer than slots here).
5. Each sequence is cut into consecutive chunks; item (b, begin, end, slot).
6. Items are ordered by length, longest first; equal lengths keep their
   generation order (b ascending, then slot).
7. ``pad_to > 0`` appends (0, 0, 0, 0) items up to that length.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Sequence, Tuple

TILE_ROWS = 128


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


@dataclass
class PlanRef:
    work: List[Tuple[int, int, int, int]] = field(default_factory=list)
    n_splits: List[int] = field(default_factory=list)
    chunk_tiles: int = 0
    slots: int = 0


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
    tiles = [max(1, _ceil_div(int(L), TILE_ROWS)) for L in seq_lens]
    longest = max(tiles)
    slots = max(1, (sm_count * ctas_per_sm) // (h_k * n_q_tiles))
    floor_chunk = max(min_chunk_tiles, _ceil_div(longest, max_splits))

    def chunks_needed(chunk: int) -> int:
        return sum(_ceil_div(t, chunk) for t in tiles)

    if force_splits > 0:
        chunk = max(floor_chunk, _ceil_div(longest, force_splits))
    elif len(tiles) >= slots or max_splits == 1:
        chunk = longest
    else:
        # Smallest chunk in [floor_chunk, longest] that fits one wave.  The
        # predicate "fits" is monotone in chunk, so bisect on it.
        left, right = floor_chunk, longest
        while left < right:
            probe = (left + right) // 2
            if chunks_needed(probe) <= slots:
                right = probe
            else:
                left = probe + 1
        chunk = left

    items = []
    n_splits = []
    for b, t in enumerate(tiles):
        k = _ceil_div(t, chunk)
        n_splits.append(k)
        for s in range(k):
            items.append((b, s * chunk, min(t, (s + 1) * chunk), s))
    # Python's sort is stable: equal lengths keep generation order.
    items = sorted(items, key=lambda it: it[1] - it[2])
    if pad_to:
        if pad_to < len(items):
            raise ValueError(f"pad_to {pad_to} < {len(items)} work items")
        items = items + [(0, 0, 0, 0)] * (pad_to - len(items))
    if max(n_splits) > max_splits:
        raise ValueError("plan exceeds max_splits")
    return PlanRef(items, n_splits, chunk, slots)

"""Pins of the plan oracle (oracle/plan_ref.py) to hand-derived plans and to
the properties the plan rule fixes.

Source: the "mjolnir/t5_decode.py" page, plan_split_kv / SplitPlan (host
helpers section).  tests/golden/plan_examples.json holds the hand
derivations.
"""

import json
import math
import os

import numpy as np
import pytest

from oracle.plan_ref import plan_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "plan_examples.json")


CASES = json.load(open(GOLDEN))["cases"]


def pin_hand_derived(fn, case):
    p = fn(**case["args"])
    assert p.chunk_tiles == case["chunk_tiles"]
    assert p.slots == case["slots"]
    assert p.n_splits == case["n_splits"]
    if "work" in case:
        assert [list(w) for w in p.work] == case["work"]
    else:
        assert len(p.work) == case["work_len"]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c["why"][:40])
def test_hand_derived_plans(case):
    pin_hand_derived(plan_ref, case)


def _check_properties(p, seq_lens, h_k, n_q_tiles, sm, cps, max_splits, force, min_chunk, pad):
    tiles = [max(1, math.ceil(L / 128)) for L in seq_lens]
    T = max(tiles)
    real = [w for w in p.work if w[2] > w[1]]
    # every tile of every sequence is covered exactly once, by contiguous chunks
    for b, t in enumerate(tiles):
        items = sorted((w for w in real if w[0] == b), key=lambda w: w[3])
        assert [w[3] for w in items] == list(range(p.n_splits[b]))
        assert items[0][1] == 0 and items[-1][2] == t
        for a, c in zip(items[:-1], items[1:]):
            assert a[2] == c[1]
        for w in items[:-1]:
            assert w[2] - w[1] == p.chunk_tiles
    assert max(p.n_splits) <= max_splits
    assert p.chunk_tiles >= max(min_chunk, math.ceil(T / max_splits))
    # longest first
    lens = [w[2] - w[1] for w in real]
    assert lens == sorted(lens, reverse=True)
    # padding
    if pad:
        assert len(p.work) == pad
        assert all(w == (0, 0, 0, 0) for w in p.work[len(real):])
    slots = max(1, sm * cps // (h_k * n_q_tiles))
    if force == 0 and (len(tiles) >= slots or max_splits == 1):
        # a batch that already fills the wave (or may not split) is not split
        assert p.chunk_tiles == T and all(n == 1 for n in p.n_splits)
    if force == 0 and len(tiles) < slots and max_splits > 1:
        total = sum(math.ceil(t / p.chunk_tiles) for t in tiles)
        lo = max(min_chunk, math.ceil(T / max_splits))
        assert total <= slots or p.chunk_tiles == lo
        # minimal: one tile smaller would not fit (or would go below the floor)
        if p.chunk_tiles > lo:
            assert sum(math.ceil(t / (p.chunk_tiles - 1)) for t in tiles) > slots


def pin_random_properties(fn, count=400):
    rng = np.random.default_rng(31)
    for _ in range(count):
        b = int(rng.integers(1, 40))
        seq_lens = rng.integers(0, 20000, size=b).tolist()
        h_k = int(rng.choice([1, 2, 8]))
        n_q_tiles = int(rng.choice([1, 2, 4]))
        sm = int(rng.choice([20, 148, 152]))
        cps = int(rng.integers(1, 5))
        max_splits = int(rng.choice([1, 16, 64, 256]))
        force = int(rng.choice([0, 0, 0, 3]))
        min_chunk = int(rng.choice([1, 1, 2]))
        p = fn(seq_lens, h_k, n_q_tiles, sm, cps, max_splits, force, min_chunk, 0)
        _check_properties(p, seq_lens, h_k, n_q_tiles, sm, cps, max_splits, force, min_chunk, 0)
        pad = len(p.work) + int(rng.integers(0, 5))
        p2 = fn(seq_lens, h_k, n_q_tiles, sm, cps, max_splits, force, min_chunk, pad)
        _check_properties(p2, seq_lens, h_k, n_q_tiles, sm, cps, max_splits, force, min_chunk, pad)


def test_random_plans_have_the_rule_properties():
    pin_random_properties(plan_ref)


def all_pins(m):
    """Every pin against module m (raises on the first that fails)."""
    for case in CASES:
        pin_hand_derived(m.plan_ref, case)
    pin_random_properties(m.plan_ref, 150)


def test_pad_below_item_count_is_rejected():
    with pytest.raises(ValueError):
        plan_ref([1000, 1000], 1, 1, 10, 1, 16, 0, 1, 1)

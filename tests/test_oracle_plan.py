"""Pins for the verification plan: closed forms, the tiny worked tree, brute-force reachability."""

import json
import os

import numpy as np
import pytest

from oracle.plan import build_plan

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiny_tree.json")


def _closure(parents):
    """Ancestor-or-self matrix by transitive closure of the parent relation (boolean powers)."""
    D = len(parents)
    A = np.eye(D, dtype=bool)
    P = np.zeros((D, D), dtype=bool)
    for v in range(1, D):
        P[v, parents[v]] = True
    R = A.copy()
    step = P.copy()
    for _ in range(D):
        R |= step
        step = (step.astype(np.int64) @ P.astype(np.int64)) > 0
    return R


def test_golden_tiny_tree():
    with open(GOLDEN) as f:
        gold = json.load(f)
    plan = build_plan(gold["parents"], gold["L"], 0, "remainder", (4,))
    assert plan.anc == [int(x, 2) for x in gold["anc_binary"]]
    assert plan.depth == gold["depth"]
    assert plan.pos == gold["pos"]
    assert plan.raw_lo == gold["raw_lo"]


def test_chain_closed_form():
    D = 40
    plan = build_plan([-1] + list(range(D - 1)), 100, 16, "window", (4,))
    assert plan.anc == [(1 << (v + 1)) - 1 for v in range(D)]
    assert plan.depth == list(range(D))


def test_star_closed_form():
    D = 64
    plan = build_plan([-1] + [0] * (D - 1), 7, 16, "window", (4,))
    assert plan.anc == [1] + [1 | (1 << v) for v in range(1, D)]
    assert plan.depth == [0] + [1] * (D - 1)


@pytest.mark.parametrize("seed", range(20))
def test_random_tree_against_reachability(seed):
    rng = np.random.default_rng(seed)
    D = int(rng.integers(1, 65))
    parents = [-1] + [int(rng.integers(0, v)) for v in range(1, D)]
    L = int(rng.integers(0, 400))
    W = int(rng.integers(1, 40))
    plan = build_plan(parents, L, W, "window", (4, 16))
    R = _closure(parents)
    for v in range(D):
        assert plan.anc[v] == sum(1 << u for u in range(D) if R[v, u])
        assert plan.depth[v] == int(R[v].sum()) - 1
        assert plan.pos[v] == L + plan.depth[v]
        assert plan.raw_lo[v] == max(0, plan.pos[v] - W)
        for m in (4, 16):
            assert plan.completes[m][v] == ((plan.pos[v] + 1) % m == 0)
            exp = sum(1 << u for u in range(D)
                      if R[v, u] and u != v and (plan.pos[u] + 1) % m == 0)
            assert plan.scr_vis[m][v] == exp


def test_remainder_tail_bounds():
    plan = build_plan([-1, 0, 1, 2, 3, 4], 253, 0, "remainder", (4,))
    # positions 253..258 -> lowest raw position = start of the unfinished 4-block
    assert plan.pos == [253, 254, 255, 256, 257, 258]
    assert plan.raw_lo == [252, 252, 252, 256, 256, 256]
    # node 2 (position 255) closes block 63; its descendants see it in the scratch pad
    assert plan.completes[4] == [False, False, True, False, False, False]
    assert plan.scr_vis[4] == [0, 0, 0, 1 << 2, 1 << 2, 1 << 2]


@pytest.mark.parametrize("bad", [[0, 0], [-1, 1], [-1, 0, 3], [-1, -1], [-1, 0, 2]])
def test_invalid_parents_rejected(bad):
    with pytest.raises(ValueError):
        build_plan(bad, 10, 4, "window", (4,))

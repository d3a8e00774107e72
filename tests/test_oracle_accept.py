"""Pins for the greedy acceptance walk: worked case, special cases, brute-force path enumeration."""

import itertools
import json
import os

import numpy as np
import pytest

from oracle.accept import accept_walk
from tree_speculative_verify_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiny_tree.json")


def _brute_force(parents, draft, target):
    """Longest root->node path whose every edge (u -> c) has draft[c] == target[u]."""
    D = len(parents)
    best = [0]
    for v in range(D):
        path = [v]
        while path[-1] != 0:
            path.append(parents[path[-1]])
        path = path[::-1]
        if all(draft[c] == target[u] for u, c in zip(path, path[1:])) and len(path) > len(best):
            best = path
    return len(best), best, int(target[best[-1]])


def test_golden_tiny():
    with open(GOLDEN) as f:
        gold = json.load(f)
    wl = workloads.tiny()
    n, path, bonus = accept_walk(gold["parents"], wl.draft[0], wl.target[0])
    assert n == gold["accept_len"]
    assert path == gold["accept_path"]
    assert bonus == int(wl.target[0][3])


def test_single_node():
    assert accept_walk([-1], [5], [9]) == (1, [0], 9)


def test_all_mismatch_and_all_match_chain():
    D = 8
    parents = [-1] + list(range(D - 1))
    draft = list(range(100, 100 + D))
    target_none = [0] * D
    assert accept_walk(parents, draft, target_none)[0] == 1
    target_all = draft[1:] + [77]
    n, path, bonus = accept_walk(parents, draft, target_all)
    assert (n, path, bonus) == (D, list(range(D)), 77)


def test_lowest_index_child_wins_a_tie():
    # two children drafting the same token: the walk takes the lower-numbered one
    n, path, _ = accept_walk([-1, 0, 0, 2], [0, 7, 7, 3], [7, 0, 3, 0])
    assert path == [0, 1]


@pytest.mark.parametrize("seed", range(30))
def test_random_trees_against_enumeration(seed):
    rng = np.random.default_rng(seed)
    D = int(rng.integers(1, 20))
    parents = [-1] + [int(rng.integers(0, v)) for v in range(1, D)]
    # distinct sibling drafts, small vocabulary so that matches happen often
    draft = [0] * D
    for u in range(D):
        kids = [c for c in range(D) if parents[c] == u]
        toks = rng.choice(6, size=len(kids), replace=False) if len(kids) <= 6 else rng.permutation(len(kids))
        for c, t in zip(kids, toks):
            draft[c] = int(t)
    target = [int(x) for x in rng.integers(0, 6, D)]
    assert accept_walk(parents, draft, target) == _brute_force(parents, draft, target)


def test_generated_trees_have_distinct_sibling_drafts():
    for wl in (workloads.small(), workloads.serving(B=8)):
        for b in range(wl.B):
            par = wl.parents[b]
            for u in range(wl.D):
                kids = [c for c in range(wl.D) if par[c] == u]
                toks = [int(wl.draft[b][c]) for c in kids]
                assert len(set(toks)) == len(toks)
            n, path, bonus = accept_walk(list(par), wl.draft[b], wl.target[b])
            assert (n, path, bonus) == _brute_force(list(par), wl.draft[b], wl.target[b])

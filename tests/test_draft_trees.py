"""Draft-side trees (CPU): the beam builder and the per-step cuts the draft-decode tests use."""

import numpy as np
import pytest

import oracle
from tree_speculative_verify_gb300 import workloads


@pytest.mark.parametrize("seed", range(5))
def test_beam_tree_levels_and_cuts(seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    par = workloads.beam_tree(rng, 2, 4)
    assert len(par) == 9 and par[0] == -1
    oracle.build_plan(par, 100, 128, "window", (4, 128))     # a valid tree (the oracle checks it)
    dep = workloads.tree_depths(par)
    # level-by-level numbering: level l holds nodes 2l-1 and 2l
    assert dep.tolist() == [0, 1, 1, 2, 2, 3, 3, 4, 4]
    for s in range(5):
        n = 1 + 2 * s
        assert all(0 <= par[v] < v for v in range(1, n))    # the cut is closed under ancestors
        assert np.all(dep[:n] <= s) and np.all(dep[n:] > s)


def test_draft_level_slices_the_inputs():
    wl = workloads.draft_beam(B=2, steps=3, L=(300, 400))
    x = workloads.draft_level(wl, 2)
    assert x.D == 5 and x.parents.shape == (2, 5) and x.Q.shape[1] == 5
    assert np.array_equal(x.parents, wl.parents[:, :5])
    assert x.rawK is wl.rawK
    with pytest.raises(ValueError):
        workloads.draft_level(workloads.serving(B=4), 2)     # pruned trees differ per request

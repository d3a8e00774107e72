"""Draft-side tree attention on the GPU: at every draft step the plan, scratch-pad and attention
calls over the tree built so far match the oracle (the same checks as a verify round, without
commit)."""

import pytest
import torch

from tree_speculative_verify_gb300 import engine, workloads
from helpers import check_round, oracle_prefix, run_oracle, upload_prefix

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("s", [1, 2, 3])
def test_draft_steps_match_oracle(s):
    base = workloads.draft_beam(B=4, steps=3, L=(1500, 2600))
    wl = workloads.draft_level(base, s)
    comp = oracle_prefix(wl)
    res = run_oracle(wl, comp, with_refresh=False)
    shape = engine.shape_for(wl)
    st = engine.alloc_state(wl)
    rb = engine.alloc_round(wl, shape)
    upload_prefix(wl, st, comp)
    st0 = st.clone()
    engine.draft_decode(shape, st, rb)
    engine.accept(shape, st, rb)        # the walk over the draft tree, for the integer checks
    torch.cuda.synchronize()
    check_round(wl, res, st0, st, rb, range(wl.B))

"""Compressed entries on the GPU: an entry committed from the scratch pad is bit-identical to the
entry prefill computes for the same committed block (both granularities, contiguous and paged),
and every prefill entry matches the oracle within the float tolerance."""

import numpy as np
import pytest
import torch

from tree_speculative_verify_gb300 import _lib, engine, workloads
from helpers import TOL, close, np32, oracle_prefix

pytestmark = pytest.mark.gpu


def _chain_workload(name, B, L, dtype="bf16", d=512, seed=5):
    # chains accepted far (high match probability) from prefixes just below a C128 boundary, so
    # the round closes C4 and C128 blocks on the accepted path
    return workloads.make_workload(name, B=B, D=12, H=4, d=d, W=128, tail_mode="window",
                                   ms=(4, 128), dtype=dtype, L=L, k=1, steps=11, p_match=0.95,
                                   seed=seed, kv_scale=0.5)


@pytest.mark.parametrize("dtype,d", [("bf16", 512), ("f32", 64), ("bf16", 128)])
def test_committed_entries_equal_prefill(dtype, d):
    wl = _chain_workload(f"commit_{dtype}_{d}", 6, [120, 121, 250, 380, 1017, 3], dtype, d)
    shape = engine.shape_for(wl)
    st = engine.alloc_state(wl)
    rb = engine.alloc_round(wl, shape)
    engine.prefill(shape, st, rb)
    engine.verify_round(shape, st, rb)
    torch.cuda.synchronize()
    assert int(rb.status.item()) == 0
    L_new = st.L.cpu().numpy()
    assert np.any(L_new // 128 > np.asarray(wl.L) // 128), "the case must commit a C128 entry"
    fresh = st.clone()
    for t in (fresh.c4K, fresh.c4V, fresh.c128K, fresh.c128V):
        t.zero_()
    engine.prefill(shape, fresh, rb)
    torch.cuda.synchronize()
    assert int(rb.status.item()) == 0
    for b in range(wl.B):
        n4, n128 = int(L_new[b]) // 4, int(L_new[b]) // 128
        assert torch.equal(st.c4K[b, :n4], fresh.c4K[b, :n4]), f"C4 K request {b}"
        assert torch.equal(st.c4V[b, :n4], fresh.c4V[b, :n4]), f"C4 V request {b}"
        assert torch.equal(st.c128K[b, :n128], fresh.c128K[b, :n128]), f"C128 K request {b}"
        assert torch.equal(st.c128V[b, :n128], fresh.c128V[b, :n128]), f"C128 V request {b}"


def test_prefill_entries_match_oracle_at_c128_edges():
    # prefixes at, just below and just above multiples of 128, and one of several thousand rows
    wl = _chain_workload("edges", 7, [0, 127, 128, 129, 255, 256, 5000])
    shape = engine.shape_for(wl)
    st = engine.alloc_state(wl)
    rb = engine.alloc_round(wl, shape)
    engine.prefill(shape, st, rb)
    torch.cuda.synchronize()
    assert int(rb.status.item()) == 0
    want = oracle_prefix(wl)
    tol = TOL[wl.dtype]
    for m, (CK, CV) in want.items():
        gk, gv = (st.c4K, st.c4V) if m == 4 else (st.c128K, st.c128V)
        for b in range(wl.B):
            n = int(wl.L[b]) // m
            close(np32(gk[b, :n]), CK[b, :n], tol, f"C{m} K request {b}")
            close(np32(gv[b, :n]), CV[b, :n], tol, f"C{m} V request {b}")

"""Page-based persistent cache on the GPU: one logical layer over three physical page pools
(raw K/V, C4, C128) sharing page ids through a page table, pages scattered over the pool.  Every
round must equal the oracle (through a logical view of the pages), and equal the contiguous cache
bit for bit (the same arithmetic reads the same values)."""

import numpy as np
import pytest
import torch

from tree_speculative_verify_gb300 import _lib, engine, workloads
from helpers import check_round, oracle_prefix, run_oracle

pytestmark = pytest.mark.gpu


def logical_view(shape, st):
    """Contiguous [B][cap][d] copies of the paged layers (test-side, for the comparisons)."""
    P, G = shape.page_tokens, shape.max_pages
    pt = st.page_table.long()

    def layer(pool):
        return pool[pt].reshape(pt.shape[0], G * pool.shape[1], pool.shape[2])
    return engine.DeviceState(rawK=layer(st.rawK), rawV=layer(st.rawV), c4K=layer(st.c4K),
                              c4V=layer(st.c4V), c128K=layer(st.c128K), c128V=layer(st.c128V),
                              L=st.L.clone())


def upload_prefix_paged(shape, st, comp):
    P = shape.page_tokens
    pt = st.page_table.cpu().numpy()
    for m, (CK, CV) in comp.items():
        dK, dV = (st.c4K, st.c4V) if m == 4 else (st.c128K, st.c128V)
        rpp = P // m
        for b in range(CK.shape[0]):
            for j0 in range(0, CK.shape[1], rpp):
                n = min(rpp, CK.shape[1] - j0)
                page = int(pt[b, j0 // rpp])
                dK[page, :n] = torch.from_numpy(CK[b, j0:j0 + n]).to(dK.dtype)
                dV[page, :n] = torch.from_numpy(CV[b, j0:j0 + n]).to(dV.dtype)


CASES = {
    "small_P512": (lambda: workloads.small(), 512, _lib.TV_ATTN_AUTO),
    "small_P1024_simt": (lambda: workloads.small(), 1024, _lib.TV_ATTN_SIMT),
    "serving_reduced_P512": (lambda: workloads.serving(B=6, L=(700, 2300)), 512, _lib.TV_ATTN_AUTO),
    "long_selection_P2048": (lambda: workloads.long_context(B=2, L=(9000, 12000), n_sel=512), 2048,
                             _lib.TV_ATTN_AUTO),
    "short_prefixes_P512": (lambda: workloads.make_workload(
        "short", B=4, D=8, H=16, d=512, W=128, tail_mode="window", ms=(4, 128), dtype="bf16",
        L=(0, 130), k=2, steps=4, p_match=0.6, seed=5, kv_scale=0.5), 512, _lib.TV_ATTN_AUTO),
    "remainder_tail_P512": (lambda: workloads.make_workload(
        "rem", B=4, D=8, H=16, d=512, W=0, tail_mode="remainder", ms=(4,), dtype="bf16",
        L=(97, 1203), k=2, steps=4, p_match=0.6, seed=13, kv_scale=0.5), 512, _lib.TV_ATTN_AUTO),
    "d64_nodes_simt_P512": (lambda: workloads.make_workload(
        "d64", B=2, D=64, H=2, d=512, W=128, tail_mode="window", ms=(4, 128), dtype="bf16",
        L=(500, 700), k=2, steps=6, p_match=0.6, seed=11, kv_scale=0.5), 512, _lib.TV_ATTN_AUTO),
    "fp32_d64_P512": (lambda: workloads.make_workload(
        "f32", B=3, D=6, H=8, d=64, W=128, tail_mode="window", ms=(4, 128), dtype="f32",
        L=(200, 900), k=2, steps=3, p_match=0.6, seed=9, kv_scale=0.5), 512, _lib.TV_ATTN_AUTO),
}


@pytest.mark.parametrize("case", list(CASES))
def test_paged_round_matches_oracle_and_contiguous(case):
    make, P, kernel = CASES[case]
    wl = make()
    comp = oracle_prefix(wl)
    res = run_oracle(wl, comp)
    # paged
    shape, st = engine.alloc_paged(wl, P, kernel)
    rb = engine.alloc_round(wl, shape)
    upload_prefix_paged(shape, st, comp)
    st0 = logical_view(shape, st)
    # the same cache contiguous, with the same capacities (so the same KV split)
    cshape = engine.shape_for(wl, kernel)
    cshape.raw_cap, cshape.c4_cap, cshape.c128_cap = shape.raw_cap, shape.c4_cap, shape.c128_cap
    cst = st0.clone()
    cst.k_idx = st.k_idx
    crb = engine.alloc_round(wl, cshape)
    engine.verify_round(shape, st, rb)
    engine.verify_round(cshape, cst, crb)
    torch.cuda.synchronize()
    check_round(wl, res, st0, logical_view(shape, st), rb, range(wl.B))
    for name in ("O", "lse", "accept_len", "path", "bonus", "committed", "scrK4", "scrK128"):
        assert torch.equal(getattr(rb, name), getattr(crb, name)), name
    view = logical_view(shape, st)
    for name in ("rawK", "rawV", "c4K", "c4V", "c128K", "c128V", "L"):
        assert torch.equal(getattr(view, name), getattr(cst, name)), name


def test_paged_prefill_matches_contiguous():
    wl = workloads.small()
    shape, st = engine.alloc_paged(wl, 512)
    rb = engine.alloc_round(wl, shape)
    engine.prefill(shape, st, rb)
    cshape = engine.shape_for(wl)
    cst = engine.alloc_state(wl)
    crb = engine.alloc_round(wl, cshape)
    engine.prefill(cshape, cst, crb)
    torch.cuda.synchronize()
    assert int(rb.status.item()) == 0
    view = logical_view(shape, st)
    for name in ("c4K", "c4V", "c128K", "c128V"):
        a, c = getattr(view, name), getattr(cst, name)
        n = min(a.shape[1], c.shape[1])
        assert torch.equal(a[:, :n], c[:, :n]), name


def test_paged_indexer_and_bad_page_id():
    wl = workloads.long_context(B=2, L=(9000, 12000), n_sel=512)
    shape, st = engine.alloc_paged(wl, 2048)
    rb = engine.alloc_round(wl, shape)
    engine.prefill(shape, st, rb)
    engine.verify_round(shape, st, rb, select=True)
    torch.cuda.synchronize()
    assert int(rb.status.item()) == 0
    # a page id outside the pool is reported; no access leaves the pool
    st.page_table[1, 0] = shape.n_pool_pages + 3
    rb.status.zero_()
    engine.verify_round(shape, st, rb, commit=False)
    torch.cuda.synchronize()
    assert int(rb.status.item()) == -1     # TV_ERR_ARG

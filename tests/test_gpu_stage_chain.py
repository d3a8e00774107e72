"""Refresh skip on the GPU (tv_shape.stage_chain = 1): tv_branch_compress stages the cached
chain's raw rows and C4 entries past the committed length, tv_refresh_commit copies only what is
left.  The visible state must equal the oracle's round, equal the unstaged path bit for bit over
several rounds, and the refresh must not read the sources of the rows it skips."""

import numpy as np
import pytest
import torch

from tree_speculative_verify_gb300 import _lib, engine, workloads
from helpers import check_round, gpu_round, oracle_prefix, run_oracle, upload_prefix

pytestmark = pytest.mark.gpu


def cached_chain(parents):
    """Root, its lowest-numbered child, that node's lowest-numbered child, ... (test side)."""
    chain = [0]
    while True:
        kids = [u for u in range(len(parents)) if parents[u] == chain[-1]]
        if not kids:
            return chain
        chain.append(min(kids))


def _edge(name, **kw):
    base = dict(B=3, D=8, H=16, d=512, W=128, tail_mode="window", ms=(4, 128), dtype="bf16",
                L=300, k=2, steps=4, p_match=0.6, seed=11, kv_scale=0.5)
    base.update(kw)
    return workloads.make_workload(name, **base)


CASES = {
    "small": lambda: workloads.small(),
    "chain24": lambda: _edge("chain24", D=24, k=1, steps=23, H=4, L=(120, 140), B=4, p_match=0.9),
    "short0": lambda: _edge("short0", L=0, seed=3),
    "short3": lambda: _edge("short3", L=3, seed=4),
    "c128_root": lambda: _edge("c128root", L=127, seed=5, p_match=0.9),
    "c128_node": lambda: _edge("c128node", L=(122, 126), B=4, D=12, k=1, steps=11, p_match=0.9),
    "c4_only": lambda: _edge("c4only", ms=(4,), L=(300, 700)),
    "c128_only": lambda: _edge("c128only", ms=(128,), L=(300, 700)),
    "f32_d64": lambda: _edge("f32_d64", d=64, H=8, dtype="f32", L=(40, 300), B=5),
    "d64_nodes": lambda: _edge("d64", D=64, k=2, steps=6, H=2, L=(500, 700), B=2, p_match=0.8),
    "serving_reduced": lambda: workloads.serving(B=6, L=(700, 2300)),
}


@pytest.mark.parametrize("case", list(CASES))
def test_staged_round_matches_oracle(case):
    wl = CASES[case]()
    comp = oracle_prefix(wl)
    res = run_oracle(wl, comp)
    shape, st0, st, rb = gpu_round(wl, comp=comp, stage_chain=1)
    check_round(wl, res, st0, st, rb, range(wl.B), staged=True)


def test_staged_refresh_reads_no_source_of_the_cached_chain():
    """Overwrite the tree K/V rows and the C4 scratch rows of the cached chain between the branch
    call and the refresh: the committed state is still the oracle's, so the refresh took those
    rows from where the branch call staged them, and read nothing of what it skipped."""
    wl = _edge("poison", D=16, k=2, steps=5, B=6, L=(250, 400), p_match=0.85, seed=17)
    comp = oracle_prefix(wl)
    res = run_oracle(wl, comp)
    shape = engine.shape_for(wl, stage_chain=1)
    st = engine.alloc_state(wl)
    rb = engine.alloc_round(wl, shape)
    upload_prefix(wl, st, comp)
    st0 = st.clone()
    engine.plan(shape, st, rb)
    engine.branch_compress(shape, st, rb)
    engine.attention(shape, st, rb)
    engine.accept(shape, st, rb)
    torch.cuda.synchronize()
    keep = [t.clone() for t in (rb.treeK, rb.treeV, rb.scrK4, rb.scrV4)]
    skipped = 0
    for b in range(wl.B):
        chain = cached_chain(wl.parents[b])
        for u in chain:
            for t in (rb.treeK, rb.treeV, rb.scrK4, rb.scrV4):
                t[b, u] = 1.0e4
        n = int(rb.accept_len[b])
        path = rb.path[b, :n].tolist()
        skipped += sum(1 for i in range(min(n, len(chain))) if path[:i + 1] == chain[:i + 1])
    assert skipped > wl.B, "the case must commit several cached-chain nodes"
    engine.refresh(shape, st, rb)
    torch.cuda.synchronize()
    for t, k in zip((rb.treeK, rb.treeV, rb.scrK4, rb.scrV4), keep):
        t.copy_(k)
    check_round(wl, res, st0, st, rb, range(wl.B), staged=True)


def _tree_inputs(wl, seed, k, steps, p_match):
    """New tree inputs (parents, tokens, Q, tree K/V) of the same sizes for a later round."""
    return workloads.make_workload("next", B=wl.B, D=wl.D, H=wl.H, d=wl.d, W=wl.W,
                                   tail_mode=wl.tail_mode, ms=wl.ms, dtype=wl.dtype, L=1, k=k,
                                   steps=steps, p_match=p_match, seed=seed, kv_scale=0.5)


def _visible_equal(a, b, L, ms, what):
    for bb in range(a.L.shape[0]):
        n = int(L[bb])
        assert torch.equal(a.rawK[bb, :n], b.rawK[bb, :n]), f"{what}: raw K request {bb}"
        assert torch.equal(a.rawV[bb, :n], b.rawV[bb, :n]), f"{what}: raw V request {bb}"
        if 4 in ms:
            assert torch.equal(a.c4K[bb, :n // 4], b.c4K[bb, :n // 4]), f"{what}: C4 K {bb}"
            assert torch.equal(a.c4V[bb, :n // 4], b.c4V[bb, :n // 4]), f"{what}: C4 V {bb}"
        if 128 in ms:
            assert torch.equal(a.c128K[bb, :n // 128], b.c128K[bb, :n // 128]), f"{what}: C128 {bb}"
            assert torch.equal(a.c128V[bb, :n // 128], b.c128V[bb, :n // 128]), f"{what}: C128 {bb}"


@pytest.mark.parametrize("kind", ["trees", "chains"])
def test_staged_rounds_equal_unstaged_bit_for_bit(kind):
    """Eight rounds from one prefix, the same inputs through both paths: every round's outputs
    (O, LSE, accept lengths, paths, committed positions) and the visible state after it are equal
    bit for bit.  Attention reads nothing past the committed length, so the staged rows there
    change none of its results.  The prefixes end near C128 boundaries so that rounds close C4
    and C128 blocks on and off the cached chain."""
    rounds = 8
    k, steps, D = (2, 4, 10) if kind == "trees" else (1, 9, 10)
    wl = _edge(f"multi_{kind}", D=D, k=k, steps=steps, B=5, L=[100, 124, 250, 380, 509],
               p_match=0.8, seed=23)
    # room for every round's rows
    extra = rounds * D + 8
    pad = torch.zeros((wl.B, extra, wl.d), dtype=wl.rawK.dtype)
    wl.rawK = torch.cat([wl.rawK, pad], 1)
    wl.rawV = torch.cat([wl.rawV, pad.clone()], 1)
    wl.raw_cap = wl.rawK.shape[1]
    wl.cap4 = wl.raw_cap // 4 + 1
    wl.cap128 = wl.raw_cap // 128 + 1
    comp = oracle_prefix(wl)
    shapes = {s: engine.shape_for(wl, stage_chain=s) for s in (0, 1)}
    states, rbs = {}, {}
    for s in (0, 1):
        states[s] = engine.alloc_state(wl)
        upload_prefix(wl, states[s], comp)
        rbs[s] = engine.alloc_round(wl, shapes[s])
    # the staged state's invisible rows start different from the unstaged state's
    states[1].rawK[:, :] = torch.where(torch.arange(wl.raw_cap)[None, :, None] >= torch.as_tensor(
        wl.L)[:, None, None], torch.full_like(wl.rawK, 7.0), wl.rawK).to(states[1].rawK.device)
    committed_chain = 0
    for r in range(rounds):
        nxt = _tree_inputs(wl, 100 + r, k, steps, 0.8)
        for s in (0, 1):
            rb = rbs[s]
            rb.parents.copy_(torch.as_tensor(nxt.parents))
            rb.draft.copy_(torch.as_tensor(nxt.draft))
            rb.target.copy_(torch.as_tensor(nxt.target))
            rb.Q.copy_(nxt.Q)
            rb.treeK.copy_(nxt.treeK)
            rb.treeV.copy_(nxt.treeV)
            engine.verify_round(shapes[s], states[s], rb)
        torch.cuda.synchronize()
        a, b = rbs[0], rbs[1]
        assert int(a.status.item()) == 0 and int(b.status.item()) == 0
        for name in ("accept_len", "path", "bonus", "committed", "O", "lse", "scrK4", "scrV4",
                     "scrK128", "scrV128"):
            assert torch.equal(getattr(a, name), getattr(b, name)), f"round {r}: {name}"
        assert torch.equal(states[0].L, states[1].L)
        L = states[0].L.cpu().numpy()
        _visible_equal(states[0], states[1], L, wl.ms, f"round {r}")
        for bb in range(wl.B):
            chain = cached_chain(nxt.parents[bb])
            n = int(a.accept_len[bb])
            path = a.path[bb, :n].tolist()
            committed_chain += sum(1 for i in range(min(n, len(chain)))
                                   if path[:i + 1] == chain[:i + 1])
    assert committed_chain > rounds * wl.B, "the rounds must commit cached-chain nodes"


def test_staged_paged_equals_unstaged_contiguous():
    """Staging through the page table: a paged staged round and a contiguous unstaged round give
    the same results and the same visible state bit for bit."""
    from test_gpu_paged import logical_view, upload_prefix_paged
    wl = workloads.serving(B=6, L=(700, 2300))
    comp = oracle_prefix(wl)
    shape, st = engine.alloc_paged(wl, 512, _lib.TV_ATTN_AUTO)
    shape.stage_chain = 1
    rb = engine.alloc_round(wl, shape)
    upload_prefix_paged(shape, st, comp)
    st0 = logical_view(shape, st)
    cshape = engine.shape_for(wl)
    cshape.raw_cap, cshape.c4_cap, cshape.c128_cap = shape.raw_cap, shape.c4_cap, shape.c128_cap
    cst = st0.clone()
    crb = engine.alloc_round(wl, cshape)
    engine.verify_round(shape, st, rb)
    engine.verify_round(cshape, cst, crb)
    torch.cuda.synchronize()
    assert int(rb.status.item()) == 0 and int(crb.status.item()) == 0
    for name in ("accept_len", "path", "committed", "O", "lse"):
        assert torch.equal(getattr(rb, name), getattr(crb, name)), name
    view = logical_view(shape, st)
    assert torch.equal(view.L, cst.L)
    _visible_equal(view, cst, cst.L.cpu().numpy(), wl.ms, "paged staged")

"""A verify round captured as a CUDA graph gives the eager round's results, replay after replay.

"Adapting Tree-Structured Speculative Decoding to DeepSeek-V4 for Efficient Inference" §4.3 replays
the verification step as a CUDA graph.  The round's five calls are captured once on fixed buffers
(with the reset of the committed lengths as a prologue, so every replay verifies the same tree
from the same prefix); every output of every replay must equal, bit for bit, what one eager round
on a copy of the same state produced: the graph runs the same kernels on the same data.  Also
covered here: page pools under the graph, and launches that may overlap their predecessor
(programmatic dependent launches) giving the results of launches one after another.
"""

import dataclasses

import pytest
import torch

from tree_speculative_verify_gb300 import _lib, engine, workloads

pytestmark = pytest.mark.gpu


def _outputs(st, rb):
    return {"O": rb.O, "lse": rb.lse, "accept_len": rb.accept_len, "path": rb.path,
            "bonus": rb.bonus, "committed": rb.committed, "anc": rb.anc, "vis4": rb.vis4,
            "vis128": rb.vis128, "scrK4": rb.scrK4, "scrK128": rb.scrK128, "L": st.L,
            "rawK": st.rawK, "rawV": st.rawV, "c4K": st.c4K, "c4V": st.c4V, "c128K": st.c128K,
            "c128V": st.c128V}


@pytest.mark.parametrize("kernel", [_lib.TV_ATTN_AUTO, _lib.TV_ATTN_SIMT])
@pytest.mark.parametrize("case", ["small", "serving_reduced"])
def test_round_graph_replays_match_eager(case, kernel):
    wl = workloads.small() if case == "small" else workloads.serving(B=8)
    shape = engine.shape_for(wl, kernel)
    st = engine.alloc_state(wl)
    rb = engine.alloc_round(wl, shape)
    engine.prefill(shape, st, rb)
    torch.cuda.synchronize()
    st_eager = st.clone()
    rb_eager = engine.alloc_round(wl, shape)
    L0 = st.L.clone()

    engine.verify_round(shape, st_eager, rb_eager)
    torch.cuda.synchronize()
    assert int(rb_eager.status.item()) == 0
    want = {k: v.clone() for k, v in _outputs(st_eager, rb_eager).items()}

    graph = engine.RoundGraph(shape, st, rb, prologue=lambda: st.L.copy_(L0, non_blocking=True))
    for _ in range(3):
        for t in (rb.O, rb.lse):
            t.fill_(float("nan"))
        for t in (rb.accept_len, rb.path, rb.bonus, rb.committed):
            t.fill_(-7)
        graph.replay()
        torch.cuda.synchronize()
        assert int(rb.status.item()) == 0
        got = _outputs(st, rb)
        for k, v in want.items():
            assert torch.equal(got[k], v), f"{k} differs after a graph replay"


def test_sparse_round_graph_with_device_indexer_matches_eager():
    # the long-context round: device indexer -> selection gather -> attention, captured once
    wl = workloads.long_context(B=2, L=(9000, 12000), n_sel=512)
    shape = engine.shape_for(wl)
    st = engine.alloc_state(wl)
    rb = engine.alloc_round(wl, shape)
    engine.prefill(shape, st, rb)
    torch.cuda.synchronize()
    st_eager = st.clone()
    rb_eager = engine.alloc_round(wl, shape)
    L0 = st.L.clone()
    engine.verify_round(shape, st_eager, rb_eager, select=True)
    torch.cuda.synchronize()
    assert int(rb_eager.status.item()) == 0
    want = {k: v.clone() for k, v in _outputs(st_eager, rb_eager).items()}
    want["sel"] = rb_eager.sel.clone()
    graph = engine.RoundGraph(shape, st, rb, select=True,
                              prologue=lambda: st.L.copy_(L0, non_blocking=True))
    for _ in range(2):
        rb.sel.fill_(-3)
        rb.O.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert int(rb.status.item()) == 0
        got = dict(_outputs(st, rb), sel=rb.sel)
        for k, v in want.items():
            assert torch.equal(got[k], v), f"{k} differs after a graph replay"


def test_paged_round_graph_matches_eager():
    # page-based pools under the captured round: the gathers of the C128 entries and raw tails
    # and the page-table addressing replay bit for bit (the eager copy shares the page table)
    wl = workloads.serving(B=6, L=(700, 2300))
    shape, st = engine.alloc_paged(wl, 512)
    rb = engine.alloc_round(wl, shape)
    engine.prefill(shape, st, rb)
    torch.cuda.synchronize()
    st_eager = st.clone()
    rb_eager = engine.alloc_round(wl, shape)
    L0 = st.L.clone()
    engine.verify_round(shape, st_eager, rb_eager)
    torch.cuda.synchronize()
    assert int(rb_eager.status.item()) == 0
    want = {k: v.clone() for k, v in _outputs(st_eager, rb_eager).items()}
    graph = engine.RoundGraph(shape, st, rb, prologue=lambda: st.L.copy_(L0, non_blocking=True))
    for _ in range(2):
        rb.O.fill_(float("nan"))
        rb.accept_len.fill_(-7)
        graph.replay()
        torch.cuda.synchronize()
        assert int(rb.status.item()) == 0
        got = _outputs(st, rb)
        for k, v in want.items():
            assert torch.equal(got[k], v), f"{k} differs after a paged graph replay"


def test_back_to_back_attention_into_one_output():
    # two attention launches in a row into the same O, lse and workspace: the second is a
    # programmatic dependent of the first and may start while the first still runs, so none of
    # its writes may come before the first has completed; the result must be the second's alone
    wl = workloads.serving(B=40, L=(1024, 4096))
    shape = engine.shape_for(wl)
    st = engine.alloc_state(wl)
    rb = engine.alloc_round(wl, shape)
    engine.prefill(shape, st, rb)
    engine.plan(shape, st, rb)
    engine.branch_compress(shape, st, rb)
    torch.cuda.synchronize()
    g = torch.Generator(device="cpu").manual_seed(11)
    Q2 = (torch.randn(rb.Q.shape, generator=g) * 0.5).to(rb.Q.dtype).to(rb.Q.device)
    rb2 = dataclasses.replace(rb, Q=Q2)   # shares O, lse, workspace and status with rb
    ref = dataclasses.replace(rb, Q=Q2, O=torch.empty_like(rb.O), lse=torch.empty_like(rb.lse),
                              workspace=torch.empty_like(rb.workspace),
                              status=torch.zeros_like(rb.status))
    engine.attention(shape, st, ref)
    torch.cuda.synchronize()
    assert int(ref.status.item()) == 0
    for _ in range(3):
        rb.O.fill_(float("nan"))
        rb.lse.fill_(float("nan"))
        engine.attention(shape, st, rb)
        engine.attention(shape, st, rb2)
        torch.cuda.synchronize()
        assert int(rb.status.item()) == 0
        assert torch.equal(rb.O, ref.O) and torch.equal(rb.lse, ref.lse)

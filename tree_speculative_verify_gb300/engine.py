"""Device buffers and the five-call verify round (allocation and marshalling only).

``DeviceState`` holds one batch's persistent cache (raw K/V, C4 and C128 entries, committed
lengths); ``RoundBuffers`` holds one round's inputs (tree, tokens, queries, tree K/V), the plan,
the scratch pad and the outputs.  ``verify_round`` enqueues tv_build_ancestor_mask,
tv_branch_compress, tv_tree_verify_attn, tv_accept_walk and tv_refresh_commit on one stream with
no host synchronisation, as "Adapting Tree-Structured Speculative Decoding to DeepSeek-V4 for
Efficient Inference" §4.1/§4.4 describe one target-verify stage.  Every step runs in the CUDA
library; PyTorch only allocates memory.
"""

import math
from dataclasses import dataclass

import torch

from . import _lib


def shape_for(wl, attn_kernel=_lib.TV_ATTN_AUTO, B=None, stage_chain=0):
    comp = 0
    if 4 in wl.ms:
        comp |= _lib.TV_COMP_C4
    if 128 in wl.ms:
        comp |= _lib.TV_COMP_C128
    return _lib.make_shape(
        B=wl.B if B is None else B, D=wl.D, H=wl.H, d=wl.d, W=wl.W,
        tail_mode=_lib.TV_TAIL_WINDOW if wl.tail_mode == "window" else _lib.TV_TAIL_REMAINDER,
        comp_mask=comp, dtype=_lib.TV_F32 if wl.dtype == "f32" else _lib.TV_BF16,
        n_sel=wl.n_sel, attn_kernel=attn_kernel, raw_cap=wl.raw_cap,
        c4_cap=wl.cap4 if 4 in wl.ms else 0, c128_cap=wl.cap128 if 128 in wl.ms else 0,
        stage_chain=stage_chain)


@dataclass
class DeviceState:
    rawK: torch.Tensor
    rawV: torch.Tensor
    c4K: torch.Tensor
    c4V: torch.Tensor
    c128K: torch.Tensor
    c128V: torch.Tensor
    L: torch.Tensor
    k_idx: torch.Tensor = None    # [B][c4_cap][64] bf16 indexer keys (sparse C4 path only)
    page_table: torch.Tensor = None   # [B][max_pages] int32 (paged pools only)

    def clone(self):
        return DeviceState(*(t.clone() for t in (self.rawK, self.rawV, self.c4K, self.c4V,
                                                 self.c128K, self.c128V, self.L)),
                           k_idx=self.k_idx, page_table=self.page_table)


@dataclass
class RoundBuffers:
    parents: torch.Tensor
    draft: torch.Tensor
    target: torch.Tensor
    Q: torch.Tensor
    treeK: torch.Tensor
    treeV: torch.Tensor
    sel: torch.Tensor
    g4: torch.Tensor
    g128: torch.Tensor
    anc: torch.Tensor
    depth: torch.Tensor
    raw_lo: torch.Tensor
    vis4: torch.Tensor
    vis128: torch.Tensor
    scrK4: torch.Tensor
    scrV4: torch.Tensor
    scrK128: torch.Tensor
    scrV128: torch.Tensor
    O: torch.Tensor
    lse: torch.Tensor
    accept_len: torch.Tensor
    path: torch.Tensor
    bonus: torch.Tensor
    committed: torch.Tensor
    status: torch.Tensor
    workspace: torch.Tensor
    q_idx: torch.Tensor = None    # [B][64] bf16 indexer queries (sparse C4 path only)
    idx_ws: torch.Tensor = None   # indexer score workspace


def alloc_state(wl, device="cuda"):
    """Persistent cache of the workload on the device: raw rows uploaded, compressed rows zero."""
    dt = wl.torch_dtype
    z = lambda n: torch.zeros((wl.B, max(n, 1), wl.d), dtype=dt, device=device)
    return DeviceState(
        rawK=wl.rawK.to(device), rawV=wl.rawV.to(device),
        c4K=z(wl.cap4 if 4 in wl.ms else 0), c4V=z(wl.cap4 if 4 in wl.ms else 0),
        c128K=z(wl.cap128 if 128 in wl.ms else 0), c128V=z(wl.cap128 if 128 in wl.ms else 0),
        L=torch.as_tensor(wl.L, dtype=torch.int32).to(device),
        k_idx=None if wl.k_idx is None else wl.k_idx.to(device))


def alloc_paged(wl, page_tokens, attn_kernel=_lib.TV_ATTN_AUTO, spare_pages=None, seed=0,
                device="cuda"):
    """Page-based persistent cache ("Adapting Tree-Structured Speculative Decoding to DeepSeek-V4
    for Efficient Inference" §4.2: one logical layer, three physical layers with shared page
    pointers).  Three pools of n_pool_pages pages -- raw K/V (P rows), C4 (P/4 entries), C128
    (P/128 entries) -- and a page table [B][max_pages] mapping each request's logical page to one
    pool page used by all three layers.  The pages of the batch are a seeded random permutation
    of the pool (a fragmented pool), plus ``spare_pages`` unused ones.  Returns (shape, state); the
    raw rows of the workload are copied into their pages, compressed entries start at zero."""
    P = int(page_tokens)
    max_pages = -(-wl.raw_cap // P)
    spare = wl.B if spare_pages is None else int(spare_pages)
    n_pool = wl.B * max_pages + spare
    perm = torch.randperm(n_pool, generator=torch.Generator().manual_seed(seed))
    table = perm[: wl.B * max_pages].reshape(wl.B, max_pages).to(torch.int32)
    dt = wl.torch_dtype
    z = lambda rows: torch.zeros((n_pool, max(rows, 1), wl.d), dtype=dt, device=device)
    rawK, rawV = z(P), z(P)
    for b in range(wl.B):
        for g in range(max_pages):
            lo, hi = g * P, min((g + 1) * P, wl.raw_cap)
            if lo < hi:
                rawK[int(table[b, g]), : hi - lo] = wl.rawK[b, lo:hi].to(device)
                rawV[int(table[b, g]), : hi - lo] = wl.rawV[b, lo:hi].to(device)
    k_idx = None
    if wl.k_idx is not None:   # indexer keys stay contiguous, one row per logical C4 entry
        k_idx = torch.zeros((wl.B, max_pages * P // 4, wl.k_idx.shape[2]), dtype=wl.k_idx.dtype,
                            device=device)
        k_idx[:, : wl.k_idx.shape[1]] = wl.k_idx.to(device)
    st = DeviceState(rawK=rawK, rawV=rawV, c4K=z(P // 4), c4V=z(P // 4), c128K=z(P // 128),
                     c128V=z(P // 128), L=torch.as_tensor(wl.L, dtype=torch.int32).to(device),
                     k_idx=k_idx, page_table=table.to(device))
    shape = shape_for(wl, attn_kernel)
    shape.raw_cap, shape.c4_cap, shape.c128_cap = max_pages * P, max_pages * P // 4, max_pages * P // 128
    shape.page_tokens, shape.max_pages, shape.n_pool_pages = P, max_pages, n_pool
    shape.page_table = st.page_table.data_ptr()
    return shape, st


def alloc_round(wl, shape, device="cuda"):
    dt = wl.torch_dtype
    B, D, H, d = wl.B, wl.D, wl.H, wl.d
    i32 = dict(dtype=torch.int32, device=device)
    i64 = dict(dtype=torch.int64, device=device)
    ws = _lib.tv_workspace_size(shape)
    g4 = wl.g[4].to(device) if 4 in wl.g else torch.zeros(d, device=device)
    g128 = wl.g[128].to(device) if 128 in wl.g else torch.zeros(d, device=device)
    sel = torch.as_tensor(wl.sel, dtype=torch.int32).to(device) if wl.sel is not None else None
    return RoundBuffers(
        parents=torch.as_tensor(wl.parents, dtype=torch.int32).to(device),
        draft=torch.as_tensor(wl.draft, dtype=torch.int32).to(device),
        target=torch.as_tensor(wl.target, dtype=torch.int32).to(device),
        Q=wl.Q.to(device), treeK=wl.treeK.to(device), treeV=wl.treeV.to(device), sel=sel,
        g4=g4, g128=g128,
        anc=torch.zeros((B, D), **i64), depth=torch.zeros((B, D), **i32),
        raw_lo=torch.zeros((B, D), **i32), vis4=torch.zeros((B, D), **i64),
        vis128=torch.zeros((B, D), **i64),
        scrK4=torch.zeros((B, D, d), dtype=dt, device=device),
        scrV4=torch.zeros((B, D, d), dtype=dt, device=device),
        scrK128=torch.zeros((B, D, d), dtype=dt, device=device),
        scrV128=torch.zeros((B, D, d), dtype=dt, device=device),
        O=torch.zeros((B, D, H, d), dtype=dt, device=device),
        lse=torch.zeros((B, D, H), dtype=torch.float32, device=device),
        accept_len=torch.zeros(B, **i32), path=torch.zeros((B, D), **i32),
        bonus=torch.zeros(B, **i32), committed=torch.zeros((B, D), **i32),
        status=torch.zeros(1, **i32),
        workspace=torch.empty(max(ws, 256), dtype=torch.uint8, device=device),
        q_idx=None if wl.q_idx is None else wl.q_idx.to(device),
        idx_ws=None if wl.q_idx is None else torch.empty(
            max(_lib.tv_indexer_workspace_size(shape), 256), dtype=torch.uint8, device=device))


def prefill(shape, st, rb, stream=None):
    _lib.tv_prefill_compress(shape, st.rawK, st.rawV, st.L, rb.g4, rb.g128, st.c4K, st.c4V,
                             st.c128K, st.c128V, rb.status, stream)


def indexer(shape, st, rb, stream=None):
    """Device selection of the n_sel C4 entries per request into ``rb.sel`` (sparse path)."""
    _lib.tv_indexer_topk(shape, 64, rb.q_idx, st.k_idx, st.L, rb.sel, rb.idx_ws, rb.status, stream)


def plan(shape, st, rb, stream=None):
    _lib.tv_build_ancestor_mask(shape, rb.parents, st.L, rb.anc, rb.depth, rb.raw_lo, rb.vis4,
                                rb.vis128, rb.status, stream)


def branch_compress(shape, st, rb, stream=None):
    _lib.tv_branch_compress(shape, st.rawK, st.rawV, st.c4K, st.c4V, st.L, rb.treeK, rb.treeV,
                            rb.parents, rb.g4, rb.g128, rb.scrK4, rb.scrV4, rb.scrK128, rb.scrV128,
                            rb.status, stream)


def attention(shape, st, rb, scale=None, stream=None):
    if scale is None:
        scale = 1.0 / math.sqrt(shape.d)
    _lib.tv_tree_verify_attn(shape, rb.Q, st.c4K, st.c4V, rb.sel, st.c128K, st.c128V, st.rawK,
                             st.rawV, st.L, rb.treeK, rb.treeV, rb.anc, rb.raw_lo, rb.vis4,
                             rb.vis128, rb.scrK4, rb.scrV4, rb.scrK128, rb.scrV128, scale, rb.O,
                             rb.lse, rb.workspace, rb.status, stream)


def accept(shape, st, rb, stream=None):
    _lib.tv_accept_walk(shape, rb.parents, rb.draft, rb.target, rb.accept_len, rb.path, rb.bonus,
                        rb.status, stream)


def refresh(shape, st, rb, stream=None):
    _lib.tv_refresh_commit(shape, rb.parents, rb.accept_len, rb.path, rb.treeK, rb.treeV,
                           rb.scrK4, rb.scrV4, rb.scrK128, rb.scrV128, st.rawK, st.rawV, st.c4K,
                           st.c4V, st.c128K, st.c128V, st.L, rb.committed, rb.status, stream)


def verify_round(shape, st, rb, scale=None, stream=None, commit=True, select=False):
    """One target-verify round: plan, scratch pad, attention, acceptance, refresh; with
    ``select`` the indexer first picks the sparse path's C4 entries on the device."""
    if select:
        indexer(shape, st, rb, stream)
    plan(shape, st, rb, stream)
    branch_compress(shape, st, rb, stream)
    attention(shape, st, rb, scale, stream)
    accept(shape, st, rb, stream)
    if commit:
        refresh(shape, st, rb, stream)


def draft_decode(shape, st, rb, scale=None, stream=None):
    """Draft-side tree attention ("Adapting Tree-Structured Speculative Decoding to DeepSeek-V4 for
    Efficient Inference" §4.1, draft decode): every candidate of the draft tree built so far
    attends to the prefix and its own ancestors, with the scratch pad isolating blocks closed
    inside the tree -- the verify round's plan, scratch-pad and attention calls on the draft
    step's tree, without acceptance or commit (nothing is accepted until the target verifies)."""
    plan(shape, st, rb, stream)
    branch_compress(shape, st, rb, stream)
    attention(shape, st, rb, scale, stream)


class RoundGraph:
    """One verify round captured as a CUDA graph on fixed buffers.

    "Adapting Tree-Structured Speculative Decoding to DeepSeek-V4 for Efficient Inference" §4.3
    replays the verification step as a CUDA graph sized for the tree configuration; here the five
    calls (and an optional ``prologue`` of stream work, e.g. refilling inputs) are captured once
    and ``replay()`` relaunches them with a single graph launch.  Construction runs one round
    without its commit (outputs and scratch pad are overwritten, the persistent state is not).
    The buffers in ``st`` / ``rb`` must stay allocated and at the same addresses; their contents
    may change between replays.
    """

    def __init__(self, shape, st, rb, scale=None, commit=True, prologue=None, select=False):
        # one eager round first, without the commit (the persistent state is left as it was):
        # the library's once-per-device set-up happens outside the capture
        verify_round(shape, st, rb, scale, None, False, select)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            stream = torch.cuda.current_stream()
            if prologue is not None:
                prologue()
            verify_round(shape, st, rb, scale, stream, commit, select)

    def replay(self):
        self.graph.replay()

"""Seeded synthetic workloads for tree-structured speculative verification.

This module only draws inputs: prefix lengths, draft trees, draft/target tokens, queries, raw K/V,
tree K/V and gate vectors.  It holds none of the verify path's arithmetic (no compression, no
masks, no attention, no acceptance), so the CUDA path and the CPU oracle can both consume exactly
the same stored inputs without sharing any of the method's code.

Conventions (from "Adapting Tree-Structured Speculative Decoding to DeepSeek-V4 for Efficient
Inference", §5.1: the budget D counts the root, ``s4_k1_d5`` is a 4-step chain of 5 verified
tokens):
* node 0 is the root (the last accepted token), ``parents[0] = -1``, ``parents[v] < v``;
* a tree configuration ``s{steps}_k{k}_d{D}`` expands a full top-k tree of ``steps`` levels below
  the root, gives the children of every node sorted U(0,1) confidences, scores a node by the
  product of confidences on its path and keeps the root plus the D-1 best nodes (ties to the node
  created first), renumbered breadth-first (an EAGLE-2-like confidence prune; the report builds
  its trees from draft confidence but gives no formula);
* ``k = 1`` gives a single chain of D nodes (linear speculation);
* draft tokens are uniform in [0, 32000) and distinct among siblings;
* target tokens stand in for the target model's greedy choices: for each node, its children are
  tried in index order and child i is matched with probability ``p_match`` (the first success
  wins); if none matches, the node's target is a token that no child drafted.

All values are drawn in fp64 from ``numpy.random.Generator(PCG64(seed))`` and rounded to the
storage dtype (fp32, or bf16 via fp32 with round-to-nearest-even).
"""

from dataclasses import dataclass, field

import numpy as np
import torch

VOCAB = 32000


@dataclass
class Workload:
    name: str
    B: int
    D: int
    H: int
    d: int
    W: int
    tail_mode: str          # "window" | "remainder"
    ms: tuple               # active compressors, e.g. (4,) or (4, 128)
    dtype: str              # "f32" | "bf16"
    L: np.ndarray           # [B] committed lengths
    raw_cap: int
    cap4: int
    cap128: int
    parents: np.ndarray     # [B, D] int32
    draft: np.ndarray       # [B, D] int32
    target: np.ndarray      # [B, D] int32
    Q: torch.Tensor         # [B, D, H, d]
    rawK: torch.Tensor      # [B, raw_cap, d], rows >= L are zero
    rawV: torch.Tensor
    treeK: torch.Tensor     # [B, D, d]
    treeV: torch.Tensor
    g: dict                 # {m: float32 tensor [d]}
    sel: np.ndarray = None  # [B, n_sel] sorted selected C4 indices, or None
    q_idx: torch.Tensor = None   # [B, 64] bf16 indexer queries (with a selection list)
    k_idx: torch.Tensor = None   # [B, cap4, 64] bf16 indexer keys of the C4 entries
    p_match: float = 0.0
    meta: dict = field(default_factory=dict)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def n_sel(self):
        return 0 if self.sel is None else int(self.sel.shape[1])


def _store(x64, dtype):
    x32 = np.ascontiguousarray(x64, dtype=np.float32)
    t = torch.from_numpy(x32)
    return t if dtype == "f32" else t.to(torch.bfloat16)


def build_tree(rng, k, steps, D):
    """Parent array of a pruned top-k draft tree (see module docstring)."""
    if D < 1:
        raise ValueError("D must be >= 1")
    if k == 1:
        return np.array([-1] + list(range(D - 1)), dtype=np.int32)
    # full tree, nodes in creation (breadth-first) order
    par, score, level = [-1], [1.0], [0]
    frontier = [0]
    for lev in range(1, steps + 1):
        nxt = []
        for u in frontier:
            conf = np.sort(rng.random(k))[::-1]
            for c in conf:
                par.append(u)
                score.append(score[u] * float(c))
                level.append(lev)
                nxt.append(len(par) - 1)
        frontier = nxt
    n_full = len(par)
    if D > n_full:
        raise ValueError(f"budget D={D} exceeds the {n_full}-node full tree")
    order = sorted(range(1, n_full), key=lambda i: (-score[i], i))
    keep = sorted([0] + order[:D - 1], key=lambda i: (level[i], i))
    new_id = {old: new for new, old in enumerate(keep)}
    parents = np.empty(D, dtype=np.int32)
    for old, new in new_id.items():
        parents[new] = -1 if old == 0 else new_id[par[old]]
    return parents


def beam_tree(rng, k, steps):
    """Parent array of a draft-side beam tree: the root's k children, then at every further level
    the k best of the k x k children of the previous level's nodes (children get sorted U(0,1)
    confidences, a node scores the product along its path; ties to the node created first).
    1 + k * steps nodes, numbered level by level."""
    parents, score = [-1], [1.0]
    frontier = [0]
    for lev in range(1, steps + 1):
        cand = []
        for u in frontier:
            for c in np.sort(rng.random(k))[::-1]:
                cand.append((u, score[u] * float(c)))
        if lev == 1:
            keep = cand
        else:
            order = sorted(range(len(cand)), key=lambda i: (-cand[i][1], i))[:k]
            keep = [cand[i] for i in sorted(order)]
        frontier = []
        for u, sc in keep:
            parents.append(u)
            score.append(sc)
            frontier.append(len(parents) - 1)
    return np.asarray(parents, dtype=np.int32)


def draw_tokens(rng, parents, p_match, forced=None):
    """Draft and target tokens of one tree (see module docstring).

    forced: optional {u: c} meaning target[u] = draft[c] (used by the tiny worked case).
    """
    D = len(parents)
    children = [[] for _ in range(D)]
    for v in range(1, D):
        children[int(parents[v])].append(v)
    draft = np.empty(D, dtype=np.int64)
    draft[0] = rng.integers(0, VOCAB)
    for u in range(D):
        if children[u]:
            toks = rng.choice(VOCAB, size=len(children[u]), replace=False)
            for c, t in zip(children[u], toks):
                draft[c] = t
    target = np.empty(D, dtype=np.int64)
    for u in range(D):
        chosen = None
        if forced is not None and u in forced:
            chosen = int(draft[forced[u]])
        elif forced is None:
            for c in children[u]:
                if rng.random() < p_match:
                    chosen = int(draft[c])
                    break
        if chosen is None:
            taken = {int(draft[c]) for c in children[u]}
            while True:
                t = int(rng.integers(0, VOCAB))
                if t not in taken:
                    break
            chosen = t
        target[u] = chosen
    return draft.astype(np.int32), target.astype(np.int32)


def _caps(L_max, D):
    raw_cap = ((L_max + 2 * D + 8 + 7) // 8) * 8
    return raw_cap, raw_cap // 4 + 1, raw_cap // 128 + 1


def make_workload(name, *, B, D, H, d, W, tail_mode, ms, dtype, L, k, steps, p_match, seed,
                  kv_scale, n_sel=0, forced=None, fixed_parents=None, beam=False):
    """Draw one workload.  ``L`` is an int (same for all requests), a (lo, hi) uniform range or a
    list of B lengths."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if isinstance(L, tuple):
        Ls = rng.integers(L[0], L[1] + 1, size=B).astype(np.int64)
    elif isinstance(L, list):
        assert len(L) == B, "one length per request"
        Ls = np.asarray(L, dtype=np.int64)
    else:
        Ls = np.full(B, int(L), dtype=np.int64)
    parents = np.empty((B, D), dtype=np.int32)
    draft = np.empty((B, D), dtype=np.int32)
    target = np.empty((B, D), dtype=np.int32)
    for b in range(B):
        if fixed_parents is not None:
            par = np.asarray(fixed_parents, dtype=np.int32)
        elif beam:
            par = beam_tree(rng, k, steps)
        else:
            par = build_tree(rng, k, steps, D)
        parents[b] = par
        draft[b], target[b] = draw_tokens(rng, par, p_match, forced)
    raw_cap, cap4, cap128 = _caps(int(Ls.max()), D)
    Q = _store(rng.standard_normal((B, D, H, d)), dtype)
    rawK = torch.zeros((B, raw_cap, d), dtype=torch.float32 if dtype == "f32" else torch.bfloat16)
    rawV = torch.zeros_like(rawK)
    for b in range(B):
        n = int(Ls[b])
        rawK[b, :n] = _store(kv_scale * rng.standard_normal((n, d)), dtype)
        rawV[b, :n] = _store(kv_scale * rng.standard_normal((n, d)), dtype)
    treeK = _store(kv_scale * rng.standard_normal((B, D, d)), dtype)
    treeV = _store(kv_scale * rng.standard_normal((B, D, d)), dtype)
    g = {m: torch.from_numpy(rng.standard_normal(d).astype(np.float32)) for m in (4, 128)}
    g = {m: g[m] for m in ms}
    sel = q_idx = k_idx = None
    if n_sel:
        # indexer inputs: a bf16 query (dim 64) per request from the root and a bf16 key per C4
        # entry; rows past a request's L // 4 entries are zero.  The selection list handed to the
        # attention tests is the stand-in of the long-context workload: the n_sel best fp64
        # scores q_idx . k_idx (ties to the lower index), sorted ascending.
        sel = np.empty((B, n_sel), dtype=np.int32)
        q_idx = torch.zeros((B, 64), dtype=torch.bfloat16)
        k_idx = torch.zeros((B, cap4, 64), dtype=torch.bfloat16)
        for b in range(B):
            n4 = int(Ls[b]) // 4
            q_idx[b] = _store(rng.standard_normal(64), "bf16")
            k_idx[b, :n4] = _store(rng.standard_normal((n4, 64)), "bf16")
            score = k_idx[b, :n4].double().numpy() @ q_idx[b].double().numpy()
            order = np.lexsort((np.arange(n4), -score))
            sel[b] = np.sort(order[:n_sel])
    return Workload(name=name, B=B, D=D, H=H, d=d, W=W, tail_mode=tail_mode, ms=tuple(ms),
                    dtype=dtype, L=Ls, raw_cap=raw_cap, cap4=cap4, cap128=cap128,
                    parents=parents, draft=draft, target=target, Q=Q, rawK=rawK, rawV=rawV,
                    treeK=treeK, treeV=treeV, g=g, sel=sel, q_idx=q_idx, k_idx=k_idx,
                    p_match=p_match,
                    meta=dict(seed=seed, k=k, steps=steps, kv_scale=kv_scale, L_spec=L))


# --- named workloads ---------------------------------------------------------------------------

def tiny(L=256, seed=0):
    """fp32, 1 request, C4 only, remainder tail, 8x1 heads, d=64, the 5-node tree
    [-1, 0, 0, 1, 2] with the target forced to accept the path 0 -> 1 -> 3."""
    return make_workload(f"tiny_fp32_L{L}", B=1, D=5, H=8, d=64, W=0, tail_mode="remainder",
                         ms=(4,), dtype="f32", L=L, k=2, steps=2, p_match=0.0, seed=seed,
                         kv_scale=1.0, forced={0: 1, 1: 3}, fixed_parents=[-1, 0, 0, 1, 2])


def small(seed=0, B=4):
    """bf16, 4 requests x 4096 prefix, C4 + C128 + 128-token window, 64x1 heads, d=512,
    top-2 tree of depth 3 pruned to D=6, child-match probability 0.6."""
    return make_workload("small_bf16", B=B, D=6, H=64, d=512, W=128, tail_mode="window",
                         ms=(4, 128), dtype="bf16", L=4096, k=2, steps=3, p_match=0.6,
                         seed=seed, kv_scale=0.5)


def serving(seed=0, B=64, D=8, L=(1024, 8192)):
    """bf16 serving batch: 64 requests, ragged prefixes U{1024..8192}, C4 + C128 + 128 window,
    64x1 heads, d=512, top-2 tree (4 draft steps) pruned to D=8, child-match probability 0.55."""
    return make_workload(f"serving_bf16_B{B}_D{D}", B=B, D=D, H=64, d=512, W=128,
                         tail_mode="window", ms=(4, 128), dtype="bf16", L=L, k=2, steps=4,
                         p_match=0.55, seed=seed, kv_scale=0.5)


def long_context(seed=0, B=8, L=(65536, 131072), n_sel=2048):
    """bf16 long context: 8 requests, prefixes U{65536..131072}, C128 entries plus the top-2048
    C4 entries of a seeded indexer score, 128 window, 64x1 heads, d=512, top-2 tree D=8, p=0.55."""
    return make_workload(f"long_bf16_B{B}", B=B, D=8, H=64, d=512, W=128, tail_mode="window",
                         ms=(4, 128), dtype="bf16", L=L, k=2, steps=4, p_match=0.55, seed=seed,
                         kv_scale=0.5, n_sel=n_sel)


def sweep_cells():
    """The budget sweep: D x batch x {chain, tree} x child-match probability, prefix 4096."""
    cells = []
    for D in (5, 6, 7, 8):
        for B in (1, 4, 16, 64):
            for kind in ("chain", "tree"):
                for p in (0.45, 0.7):
                    cells.append(dict(D=D, B=B, kind=kind, p=p))
    return cells


def sweep_cell(idx, D, B, kind, p, L=4096):
    k, steps = (1, D - 1) if kind == "chain" else (2, 4)
    return make_workload(f"sweep_{kind}_D{D}_B{B}_p{p}", B=B, D=D, H=64, d=512, W=128,
                         tail_mode="window", ms=(4, 128), dtype="bf16", L=L, k=k, steps=steps,
                         p_match=p, seed=1000 + idx, kv_scale=0.5)


def tree_depths(parents):
    """Depth of every node of one parent array (root 0)."""
    dep = np.zeros(len(parents), dtype=np.int64)
    for v in range(1, len(parents)):
        dep[v] = dep[int(parents[v])] + 1
    return dep


def draft_beam(seed=0, B=64, steps=3, L=(1024, 8192)):
    """Draft-decode workload: the serving batch's cache geometry (C4 + C128 + 128 window, 64x1
    heads, d = 512, bf16) with a width-2 beam tree of ``steps`` draft levels per request
    (D = 1 + 2 * steps); ``draft_level`` cuts it to the tree the draft model attends over at each
    step."""
    return make_workload(f"draft_beam_B{B}_s{steps}", B=B, D=1 + 2 * steps, H=64, d=512, W=128,
                         tail_mode="window", ms=(4, 128), dtype="bf16", L=L, k=2, steps=steps,
                         p_match=0.55, seed=seed, kv_scale=0.5, beam=True)


def draft_level(wl, s):
    """The draft-decode view of a workload at draft step ``s``: every request's tree cut to its
    nodes of depth <= s.  Nodes are numbered level by level, so these are the first D_s nodes; the
    cut needs every request to have the same D_s (true of beam trees).  Queries, tree K/V and
    tokens are sliced; the caches are shared."""
    deps = [tree_depths(wl.parents[b]) for b in range(wl.B)]
    counts = {int((d <= s).sum()) for d in deps}
    if len(counts) != 1:
        raise ValueError(f"requests have different node counts at depth <= {s}: {sorted(counts)}")
    Ds = counts.pop()
    cut = lambda a: np.ascontiguousarray(a[:, :Ds])
    tcut = lambda t: t[:, :Ds].contiguous()
    return Workload(name=f"{wl.name}_draft{s}", B=wl.B, D=Ds, H=wl.H, d=wl.d, W=wl.W,
                    tail_mode=wl.tail_mode, ms=wl.ms, dtype=wl.dtype, L=wl.L, raw_cap=wl.raw_cap,
                    cap4=wl.cap4, cap128=wl.cap128, parents=cut(wl.parents), draft=cut(wl.draft),
                    target=cut(wl.target), Q=tcut(wl.Q), rawK=wl.rawK, rawV=wl.rawV,
                    treeK=tcut(wl.treeK), treeV=tcut(wl.treeV), g=wl.g, sel=wl.sel,
                    q_idx=wl.q_idx, k_idx=wl.k_idx, p_match=wl.p_match,
                    meta=dict(wl.meta, draft_step=s))

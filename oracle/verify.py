"""Branch-aware causal tree-verify attention (oracle; test infrastructure only).

[TSD-V4] §3.1: every candidate attends to the accepted context and to its own ancestors, never to
other branches.  [TSD-V4] §3.2 and §4.2: blocks that a branch completes are compressed for that
branch alone, into a scratch pad, and never written to the persistent cache during verification.

Semantics fixed here (the report is silent on the details; these are the plainest readings):

* a query at position p sees
  - compressed entry (m, j) iff its block ends strictly before p: ``m*j + m - 1 <= p - 1``;
  - raw tokens at positions ``raw_lo(p) .. p`` (itself included);
* for tree node v the sequence is ``prefix (positions < L) + tokens of the path root -> v``, so v
  sees: the persistent C4 / C128 entries (all of them end at or before L - 1 <= pos[v] - 1; for C4
  only the selected ones when a selection list is given), the scratch entries of its proper
  ancestors that close a block, the raw prefix positions ``raw_lo[v] .. L-1`` and the
  ancestor-or-self tree tokens at positions ``>= raw_lo[v]``;
* logit ``l = (q . k) / sqrt(d)``; softmax over the visible set; ``O = sum p_j v_j``;
  ``LSE = ln sum_j exp(l_j)``.  H query heads share the single K/V head.

Node v therefore computes exactly what ordinary causal decoding computes at position pos[v] of the
linear sequence prefix + path(v); the self-tests check this against brute force.
"""

import math
from dataclasses import dataclass

import numpy as np

from .compress import gated_block_sum
from .plan import build_plan
from .storage import round_to_storage, to_f64


@dataclass(frozen=True)
class VerifyConfig:
    """Static description of one workload.

    ms: active compressors, e.g. (4,) or (4, 128); W: raw window (tail_mode "window");
    tail_mode: "window" | "remainder"; store: storage dtype of compressed entries
    ("bf16", "f32" or "f64" for the unrounded self-checks).
    """

    H: int
    d: int
    ms: tuple
    W: int
    tail_mode: str
    store: str


def path_to_root(parents, v):
    """Nodes on the path root -> v, in order (root first)."""
    path = [v]
    while path[-1] != 0:
        path.append(int(parents[path[-1]]))
    return path[::-1]


def sequence_row(pos, L, path, raw, tree):
    """Row at sequence position ``pos`` of prefix + path: raw prefix below L, the path's node above."""
    if pos < L:
        return to_f64(raw[pos])
    return to_f64(tree[path[pos - L]])


def scratch_entries(cfg, parents, L, rawK, rawV, treeK, treeV, g, plan=None):
    """Scratch-pad entries of one request.

    Returns {(m, u): (CK, CV)} for every node u whose token closes a block of compressor m; the
    block is read from the sequence prefix + path(u) and the entry is rounded to storage.
    """
    if plan is None:
        plan = build_plan(parents, L, cfg.W, cfg.tail_mode, cfg.ms)
    out = {}
    for m in cfg.ms:
        for u in range(len(parents)):
            if not plan.completes[m][u]:
                continue
            path = path_to_root(parents, u)
            end = plan.pos[u]
            Kb = np.stack([sequence_row(t, L, path, rawK, treeK) for t in range(end + 1 - m, end + 1)])
            Vb = np.stack([sequence_row(t, L, path, rawV, treeV) for t in range(end + 1 - m, end + 1)])
            ck, cv = gated_block_sum(Kb, Vb, g[m])
            out[(m, u)] = (round_to_storage(ck, cfg.store), round_to_storage(cv, cfg.store))
    return out


def visible_set(cfg, v, plan, L, comp, sel, rawK, rawV, treeK, treeV, scratch):
    """(Kvis, Vvis) of node v: every row v attends to, as fp64 [N, d] arrays.

    comp: {m: (CK, CV)} persistent entries of this request (rows 0 .. L//m - 1 are valid);
    sel: None, or the selected C4 entry indices; scratch: output of ``scratch_entries``.
    """
    rowsK, rowsV = [], []
    for m in cfg.ms:
        CK, CV = comp[m]
        n = L // m
        idx = range(n)
        if m == 4 and sel is not None:
            idx = [int(j) for j in sel]
        for j in idx:
            rowsK.append(to_f64(CK[j]))
            rowsV.append(to_f64(CV[j]))
    for m in cfg.ms:
        for u in range(len(plan.anc)):
            if (plan.scr_vis[m][v] >> u) & 1:
                ck, cv = scratch[(m, u)]
                rowsK.append(ck)
                rowsV.append(cv)
    for t in range(plan.raw_lo[v], L):
        rowsK.append(to_f64(rawK[t]))
        rowsV.append(to_f64(rawV[t]))
    for u in range(len(plan.anc)):
        if (plan.anc[v] >> u) & 1 and plan.pos[u] >= plan.raw_lo[v]:
            rowsK.append(to_f64(treeK[u]))
            rowsV.append(to_f64(treeV[u]))
    return np.stack(rowsK), np.stack(rowsV)


def attend(Qv, Kvis, Vvis):
    """Softmax attention of H query rows over one visible set: returns O [H, d], LSE [H]."""
    d = Qv.shape[-1]
    S = (to_f64(Qv) @ Kvis.T) / math.sqrt(d)
    M = S.max(axis=1, keepdims=True)
    E = np.exp(S - M)
    Z = E.sum(axis=1, keepdims=True)
    O = (E @ Vvis) / Z
    LSE = (M + np.log(Z))[:, 0]
    return O, LSE


def tree_verify_attn_request(cfg, parents, L, Q, comp, sel, rawK, rawV, treeK, treeV, g):
    """Verify attention of one request: O [D, H, d] and LSE [D, H] in fp64, plus the scratch pad.

    Q: [D, H, d] queries of the tree nodes; other arguments as in ``visible_set`` /
    ``scratch_entries``.
    """
    plan = build_plan(parents, L, cfg.W, cfg.tail_mode, cfg.ms)
    scratch = scratch_entries(cfg, parents, L, rawK, rawV, treeK, treeV, g, plan)
    D = len(parents)
    O = np.zeros((D, cfg.H, cfg.d))
    LSE = np.zeros((D, cfg.H))
    for v in range(D):
        Kvis, Vvis = visible_set(cfg, v, plan, L, comp, sel, rawK, rawV, treeK, treeV, scratch)
        O[v], LSE[v] = attend(Q[v], Kvis, Vvis)
    return O, LSE, scratch, plan

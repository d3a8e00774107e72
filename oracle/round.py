"""One full target-verify round over a batch (oracle; test infrastructure only).

[TSD-V4] §4.1 and §4.4: verify preprocess (the plan) -> target verify with scratch-pad isolation
-> accepted-path selection -> accepted-path state refresh.  The target model's own token choice
is an input here (``target``): this library verifies given queries and tokens, it holds no model.

Requests are independent; the oracle processes them one at a time, each in fp64 copies of its own
state, so memory stays bounded at the longest-context workloads.
"""

import numpy as np

from .accept import accept_walk
from .refresh import refresh_commit_request
from .storage import to_f64
from .verify import tree_verify_attn_request


def verify_round(cfg, parents, L, Q, comp, sel, rawK, rawV, treeK, treeV, g, draft, target,
                 requests=None, with_refresh=True):
    """Run the five steps for the listed requests (all by default).

    Array arguments are indexed by request first: parents/draft/target [B, D], L [B],
    Q [B, D, H, d], rawK/rawV [B, cap, d], treeK/treeV [B, D, d], comp {m: (CK, CV)} with
    CK/CV [B, cap_m, d], sel None or [B, n_sel], g {m: [d]}.

    Returns {b: result} where result holds the plan, O [D, H, d], LSE [D, H], the scratch pad
    {(m, u): (CK, CV)}, the walk (accept_len, path, bonus) and, with ``with_refresh``, the new
    length, the committed positions, the raw rows written and the compressed entries written.
    """
    B = len(L)
    if requests is None:
        requests = range(B)
    out = {}
    for b in requests:
        Lb = int(L[b])
        par = [int(x) for x in parents[b]]
        D = len(par)
        comp_b = {m: (comp[m][0][b], comp[m][1][b]) for m in cfg.ms}
        sel_b = None if sel is None else sel[b]
        O, LSE, scratch, plan = tree_verify_attn_request(
            cfg, par, Lb, Q[b], comp_b, sel_b, rawK[b], rawV[b], treeK[b], treeV[b], g)
        n, path, bonus = accept_walk(par, draft[b], target[b])
        res = dict(plan=plan, O=O, LSE=LSE, scratch=scratch, accept_len=n, path=path, bonus=bonus)
        if with_refresh:
            hi = Lb + n
            rK = to_f64(rawK[b][:hi]).copy()
            rV = to_f64(rawV[b][:hi]).copy()
            cK = {}
            for m in cfg.ms:
                j_hi = hi // m + 1
                cK[m] = (to_f64(comp[m][0][b][:j_hi]).copy(), to_f64(comp[m][1][b][:j_hi]).copy())
            # the refresh only writes rows >= L and entries of blocks ending at >= L
            L_new, committed = refresh_commit_request(
                cfg.ms, cfg.store, Lb, path, D, treeK[b], treeV[b], g, rK, rV, cK)
            written_entries = {}
            for m in cfg.ms:
                for e in range(Lb, L_new):
                    if (e + 1) % m == 0:
                        j = (e + 1) // m - 1
                        written_entries[(m, j)] = (cK[m][0][j].copy(), cK[m][1][j].copy())
            res.update(L_new=L_new, committed=committed,
                       raw_rows=(rK[Lb:L_new].copy(), rV[Lb:L_new].copy()),
                       entries=written_entries)
        out[b] = res
    return out

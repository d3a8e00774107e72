"""Accepted-path state refresh (oracle; test infrastructure only).

[TSD-V4] §3.2 and §4.2: once the accepted path is known, the token history, the raw (sliding-window)
KV and the CSA/HCA compressed states are refreshed so that they all describe the same logical
prefix; nothing from a rejected branch reaches the persistent state.

For an accepted path of n nodes (root included) of a request with committed length L:
* raw K/V rows ``L + i`` <- the tree K/V of ``path[i]`` (exact copies), i < n;
* for every compressor m and every position e in ``[L, L + n - 1]`` with ``(e + 1) % m == 0``,
  entry ``(e + 1) / m - 1`` <- the gated sum of the now-committed raw rows ``e + 1 - m .. e``;
* ``L <- L + n``; the committed position of path node i is ``L_old + i`` (-1 beyond n).
"""

import numpy as np

from .compress import gated_block_sum
from .storage import round_to_storage, to_f64


def refresh_commit_request(ms, store, L, path, D, treeK, treeV, g, rawK, rawV, comp):
    """Commit one request's accepted path, in place on fp64 copies of its state.

    rawK, rawV: [cap, d] fp64 arrays; comp: {m: (CK, CV)} fp64 arrays; returns
    (L_new, committed_pos[D]).
    """
    n = len(path)
    if L + n > rawK.shape[0]:
        raise ValueError("raw capacity exceeded")
    for i, u in enumerate(path):
        rawK[L + i] = to_f64(treeK[u])
        rawV[L + i] = to_f64(treeV[u])
    for m in ms:
        CK, CV = comp[m]
        for e in range(L, L + n):
            if (e + 1) % m != 0:
                continue
            j = (e + 1) // m - 1
            if j >= CK.shape[0]:
                raise ValueError("compressed capacity exceeded")
            ck, cv = gated_block_sum(rawK[e + 1 - m:e + 1], rawV[e + 1 - m:e + 1], g[m])
            CK[j] = round_to_storage(ck, store)
            CV[j] = round_to_storage(cv, store)
    committed = [L + i for i in range(n)] + [-1] * (D - n)
    return L + n, np.array(committed, dtype=np.int64)

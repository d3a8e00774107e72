"""The online sequence compressor, C4 and C128 (oracle; test infrastructure only).

[TSD-V4] §2.2 says CSA and HCA build compressed context representations online along the
sequence, at different granularities, but gives no formula.  This library fixes one concrete
stand-in and keeps to it everywhere:

* compressor ``m`` (m = 4 for C4, m = 128 for C128) cuts positions into blocks
  ``[m*j, m*j + m - 1]``; block ``j`` becomes compressed entry ``j`` once all ``m`` of its
  tokens exist;
* the gate logit of token ``t`` in the block is ``z_t = K_t . g_m`` (plain dot product with the
  compressor's gate vector, no scale);
* the gate weights are ``w = softmax(z)`` over the ``m`` tokens of the block (max subtracted);
* the entry is ``C_K = sum_t w_t K_t`` and ``C_V = sum_t w_t V_t`` (one weight vector for both).

C4 and C128 read the raw tokens independently of each other.
"""

import numpy as np

from .storage import round_to_storage, to_f64


def gated_block_sum(Kb, Vb, g):
    """Compressed (C_K, C_V) of one block.

    Kb, Vb: [m, d] raw keys / values of the block's tokens in position order; g: [d].
    Returns two fp64 vectors of length d (unrounded).
    """
    Kb = to_f64(Kb)
    Vb = to_f64(Vb)
    g = to_f64(g)
    z = Kb @ g
    w = np.exp(z - z.max())
    w = w / w.sum()
    return w @ Kb, w @ Vb


def compress_blocks(rawK, rawV, j0, j1, m, g, store):
    """Entries ``j0 <= j < j1`` of compressor ``m`` from one request's raw K/V rows.

    rawK, rawV: [>= m*j1, d].  Returns (CK, CV), each [j1 - j0, d], rounded to ``store``.
    Each entry is ``gated_block_sum`` of its own block; rows are widened to fp64 slab by slab
    only to bound memory.
    """
    d = rawK.shape[1]
    n = j1 - j0
    CK = np.empty((n, d), dtype=np.float64)
    CV = np.empty((n, d), dtype=np.float64)
    slab = max(1, (1 << 14) // m)
    for s0 in range(0, n, slab):
        s1 = min(n, s0 + slab)
        r0 = m * (j0 + s0)
        Kslab = to_f64(rawK[r0:m * (j0 + s1)])
        Vslab = to_f64(rawV[r0:m * (j0 + s1)])
        for j in range(s0, s1):
            t0 = m * (j - s0)
            CK[j], CV[j] = gated_block_sum(Kslab[t0:t0 + m], Vslab[t0:t0 + m], g)
    return round_to_storage(CK, store), round_to_storage(CV, store)


def compress_prefix(rawK, rawV, L, m, g, store):
    """All complete blocks of a committed prefix of length ``L``: entries ``0 <= j < L // m``."""
    return compress_blocks(rawK, rawV, 0, L // m, m, g, store)

"""Indexer top-k selection of persistent C4 entries (oracle; test infrastructure only).

The report's compressed attention is "Compressed Sparse Attention" ([TSD-V4] §2.2): a query does
not attend to every compressed C4 entry of a long prefix but to a selected subset.  The report
gives no selection rule; the long-context workload fixes a stand-in: an indexer key k_idx[j]
(dimension d_idx = 64) per persistent C4 entry j and an indexer query q_idx per request (from the
root query); entry j scores q_idx . k_idx[j]; the n_sel best entries are kept, equal scores going
to the lower index, and the list is handed to attention in ascending order.

Precision (the scores decide an integer selection, so both sides take that decision in one
precision): q_idx and k_idx are stored bf16; the score is the fp32 sum of the d_idx products in
index order i = 0, 1, ..., d_idx - 1, each product and each partial sum rounded to fp32 with
round-to-nearest-even and no fused multiply-add.  (A product of two bf16 values is exact in fp32,
so only the additions round.)
"""

import numpy as np


def index_scores(q_idx, k_idx):
    """Scores of the C4 entries of one request.

    q_idx: [d_idx] and k_idx: [n4, d_idx], values exactly representable in bf16 (any float dtype).
    Returns float32 [n4]: sequential fp32 sums in index order.
    """
    q = np.asarray(q_idx, dtype=np.float32)
    K = np.asarray(k_idx, dtype=np.float32)
    s = np.zeros(K.shape[0], dtype=np.float32)
    for i in range(q.shape[0]):
        prod = (K[:, i] * q[i]).astype(np.float32)       # exact for bf16 operands
        s = (s + prod).astype(np.float32)                 # one fp32 rounding per term
    return s


def topk_ascending(scores, k):
    """The k best entries (largest score first, equal scores: lower index first), returned as
    an ascending int32 index list.  k must not exceed the number of entries."""
    scores = np.asarray(scores)
    n = scores.shape[0]
    if k > n:
        raise ValueError(f"k = {k} exceeds the {n} entries")
    # primary key: score, descending; secondary: index, ascending
    order = sorted(range(n), key=lambda j: (-float(scores[j]), j))
    return np.sort(np.asarray(order[:k], dtype=np.int32))


def indexer_select(q_idx, k_idx, L, k):
    """Selection list of one request with committed length L: the top k of its L // 4 C4 entries."""
    n4 = int(L) // 4
    return topk_ascending(index_scores(q_idx, np.asarray(k_idx)[:n4]), k)

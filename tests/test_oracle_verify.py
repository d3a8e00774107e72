"""Checks (a) and (b) plus special cases: the oracle's tree verify against brute-force decoding.

(a) every tree node's output equals ordinary causal decoding at its position of the LINEAR
    sequence prefix + path(root -> node), with every compressed entry rebuilt from scratch;
(b) a top-1 chain verified in one pass equals decoding its tokens one at a time, committing each
    token through the oracle's refresh before decoding the next.

The brute force below shares nothing with the oracle's tree logic: it builds the linear sequence,
recompresses each block with its own loops, and attends with explicit per-head loops.
"""

import math

import numpy as np
import pytest
from scipy.special import logsumexp

from oracle import (VerifyConfig, accept_walk, build_plan, compress_prefix, refresh_commit_request,
                    tree_verify_attn_request)


def _bf_block(seqK, seqV, lo, hi, g):
    z = [float(np.dot(seqK[t], g)) for t in range(lo, hi)]
    zm = max(z)
    w = [math.exp(x - zm) for x in z]
    s = sum(w)
    ck = sum((wt / s) * seqK[t] for wt, t in zip(w, range(lo, hi)))
    cv = sum((wt / s) * seqV[t] for wt, t in zip(w, range(lo, hi)))
    return ck, cv


def linear_decode(seqK, seqV, p, q, ms, g, W, tail_mode):
    """Causal decode of the query at position p of a linear sequence (positions 0..p)."""
    keys, vals = [], []
    for m in ms:
        j = 0
        while m * j + m - 1 <= p - 1:
            ck, cv = _bf_block(seqK, seqV, m * j, m * j + m, g[m])
            keys.append(ck)
            vals.append(cv)
            j += 1
    lo = max(0, p - W) if tail_mode == "window" else min(ms) * (p // min(ms))
    for t in range(lo, p + 1):
        keys.append(seqK[t])
        vals.append(seqV[t])
    H, d = q.shape
    O = np.zeros((H, d))
    LSE = np.zeros(H)
    for h in range(H):
        logits = np.array([float(np.dot(q[h], k)) / math.sqrt(d) for k in keys])
        mx = logits.max()
        w = np.exp(logits - mx)
        O[h] = sum(wi * vi for wi, vi in zip(w, vals)) / w.sum()
        LSE[h] = mx + math.log(w.sum())
    return O, LSE


def _random_case(rng, D, L, d, H, ms, kv_scale=1.0, cap_extra=40):
    parents = [-1] + [int(rng.integers(0, v)) for v in range(1, D)]
    cap = L + cap_extra
    rawK = np.zeros((cap, d))
    rawV = np.zeros((cap, d))
    rawK[:L] = rng.standard_normal((L, d)) * kv_scale
    rawV[:L] = rng.standard_normal((L, d)) * kv_scale
    treeK = rng.standard_normal((D, d)) * kv_scale
    treeV = rng.standard_normal((D, d)) * kv_scale
    Q = rng.standard_normal((D, H, d))
    g = {m: rng.standard_normal(d) * 0.5 for m in ms}
    return parents, rawK, rawV, treeK, treeV, Q, g


CASES = [
    # (tail_mode, W, ms, L, D)
    ("window", 8, (4, 16), 37, 9),
    ("window", 8, (4, 16), 61, 12),
    ("window", 5, (4, 8), 3, 7),
    ("remainder", 0, (4,), 253, 6),
    ("remainder", 0, (4,), 254, 5),
    ("remainder", 0, (4, 16), 45, 10),
    ("window", 128, (4, 128), 250, 8),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_check_a_every_node_equals_linear_decode(case):
    tail_mode, W, ms, L, D = CASES[case]
    rng = np.random.default_rng(100 + case)
    d, H = 8, 3
    parents, rawK, rawV, treeK, treeV, Q, g = _random_case(rng, D, L, d, H, ms)
    cfg = VerifyConfig(H=H, d=d, ms=ms, W=W, tail_mode=tail_mode, store="f64")
    comp = {m: compress_prefix(rawK, rawV, L, m, g[m], "f64") for m in ms}
    O, LSE, scratch, plan = tree_verify_attn_request(cfg, parents, L, Q, comp, None,
                                                     rawK, rawV, treeK, treeV, g)
    n_scratch = sum(1 for m in ms for u in range(D) if plan.completes[m][u])
    assert len(scratch) == n_scratch
    for v in range(D):
        path = [v]
        while path[-1] != 0:
            path.append(parents[path[-1]])
        path = path[::-1]
        seqK = np.concatenate([rawK[:L], treeK[path]])
        seqV = np.concatenate([rawV[:L], treeV[path]])
        p = L + len(path) - 1
        Ob, LSEb = linear_decode(seqK, seqV, p, Q[v], ms, g, W, tail_mode)
        np.testing.assert_allclose(O[v], Ob, rtol=0, atol=1e-12)
        np.testing.assert_allclose(LSE[v], LSEb, rtol=0, atol=1e-12)


def test_scratch_pad_is_exercised():
    """The cases above include nodes that close blocks of both compressors."""
    seen = set()
    for tail_mode, W, ms, L, D in CASES:
        rng = np.random.default_rng(0)
        parents = [-1] + list(range(D - 1))
        plan = build_plan(parents, L, W, tail_mode, ms)
        for m in ms:
            if any(plan.completes[m]):
                seen.add(m)
    assert {4, 16, 128} <= seen


@pytest.mark.parametrize("store", ["bf16", "f64"])
def test_check_b_chain_equals_sequential_decode_with_commits(store):
    rng = np.random.default_rng(7)
    D, L, d, H, W, ms = 9, 121, 16, 2, 6, (4, 8)
    _, rawK, rawV, treeK, treeV, Q, g = _random_case(rng, D, L, d, H, ms, cap_extra=2 * D)
    if store == "bf16":
        from oracle.storage import round_to_storage
        rawK, rawV, treeK, treeV = (round_to_storage(x, "bf16") for x in (rawK, rawV, treeK, treeV))
    chain = [-1] + list(range(D - 1))
    cfg = VerifyConfig(H=H, d=d, ms=ms, W=W, tail_mode="window", store=store)
    comp = {m: compress_prefix(rawK, rawV, L, m, g[m], store) for m in ms}
    O, LSE, _, _ = tree_verify_attn_request(cfg, chain, L, Q, comp, None, rawK, rawV, treeK, treeV, g)
    # sequential: a one-node tree per token, committed before the next one is decoded
    sK, sV = rawK.copy(), rawV.copy()
    cap_m = {m: (L + D) // m + 1 for m in ms}
    scomp = {}
    for m in ms:
        ck = np.zeros((cap_m[m], d))
        cv = np.zeros((cap_m[m], d))
        ck[:L // m], cv[:L // m] = comp[m]
        scomp[m] = (ck, cv)
    Lc = L
    for t in range(D):
        Ot, LSEt, _, _ = tree_verify_attn_request(cfg, [-1], Lc, Q[t:t + 1], scomp, None,
                                                   sK, sV, treeK[t:t + 1], treeV[t:t + 1], g)
        np.testing.assert_allclose(Ot[0], O[t], rtol=0, atol=1e-12)
        np.testing.assert_allclose(LSEt[0], LSE[t], rtol=0, atol=1e-12)
        n, path, _ = accept_walk([-1], [0], [0])
        Lc, _ = refresh_commit_request(ms, store, Lc, path, 1, treeK[t:t + 1], treeV[t:t + 1], g,
                                       sK, sV, scomp)
    assert Lc == L + D


def test_single_visible_entry_returns_its_value():
    rng = np.random.default_rng(11)
    d, H = 8, 4
    cfg = VerifyConfig(H=H, d=d, ms=(4,), W=0, tail_mode="remainder", store="f64")
    treeK = rng.standard_normal((1, d))
    treeV = rng.standard_normal((1, d))
    Q = rng.standard_normal((1, H, d))
    raw = np.zeros((4, d))
    comp = {4: (np.zeros((1, d)), np.zeros((1, d)))}
    O, LSE, _, _ = tree_verify_attn_request(cfg, [-1], 0, Q, comp, None, raw, raw, treeK, treeV,
                                            {4: np.zeros(d)})
    for h in range(H):
        np.testing.assert_allclose(O[0, h], treeV[0], atol=1e-15)
        assert abs(LSE[0, h] - float(Q[0, h] @ treeK[0]) / math.sqrt(d)) < 1e-13


def test_zero_query_gives_mean_of_visible_values_and_lse_is_logsumexp():
    rng = np.random.default_rng(12)
    d, H, L, W, D = 8, 2, 30, 6, 4
    parents, rawK, rawV, treeK, treeV, Q, g = _random_case(rng, D, L, d, H, (4,))
    cfg = VerifyConfig(H=H, d=d, ms=(4,), W=W, tail_mode="window", store="f64")
    comp = {4: compress_prefix(rawK, rawV, L, 4, g[4], "f64")}
    Q0 = np.zeros_like(Q)
    O, LSE, scratch, plan = tree_verify_attn_request(cfg, parents, L, Q0, comp, None,
                                                     rawK, rawV, treeK, treeV, g)
    O1, LSE1, _, _ = tree_verify_attn_request(cfg, parents, L, Q, comp, None,
                                              rawK, rawV, treeK, treeV, g)
    for v in range(D):
        # visible set size: L//4 compressed + scratch of proper ancestors + window raw + path tokens
        n_raw = L - plan.raw_lo[v]
        n_tree = bin(plan.anc[v]).count("1")
        n_scr = bin(plan.scr_vis[4][v]).count("1")
        N = L // 4 + n_scr + n_raw + n_tree
        vis_v = list(comp[4][1]) + [scratch[(4, u)][1] for u in range(D) if (plan.scr_vis[4][v] >> u) & 1] \
            + list(rawV[plan.raw_lo[v]:L]) + [treeV[u] for u in range(D) if (plan.anc[v] >> u) & 1]
        assert len(vis_v) == N
        np.testing.assert_allclose(O[v, 0], np.mean(vis_v, axis=0), atol=1e-14)
        assert abs(LSE[v, 0] - math.log(N)) < 1e-13
        vis_k = list(comp[4][0]) + [scratch[(4, u)][0] for u in range(D) if (plan.scr_vis[4][v] >> u) & 1] \
            + list(rawK[plan.raw_lo[v]:L]) + [treeK[u] for u in range(D) if (plan.anc[v] >> u) & 1]
        for h in range(H):
            logits = np.array([Q[v, h] @ k for k in vis_k]) / math.sqrt(d)
            assert abs(LSE1[v, h] - logsumexp(logits)) < 1e-12


def test_selection_list_restricts_persistent_c4_only():
    rng = np.random.default_rng(13)
    d, H, L, W, D = 8, 2, 64, 8, 5
    parents, rawK, rawV, treeK, treeV, Q, g = _random_case(rng, D, L, d, H, (4, 16))
    cfg = VerifyConfig(H=H, d=d, ms=(4, 16), W=W, tail_mode="window", store="f64")
    comp = {m: compress_prefix(rawK, rawV, L, m, g[m], "f64") for m in (4, 16)}
    sel = np.array([1, 5, 6, 15])
    # dropping unselected C4 entries is the same as zeroing their probability: rebuild by hand
    O, _, _, _ = tree_verify_attn_request(cfg, parents, L, Q, comp, sel, rawK, rawV, treeK, treeV, g)
    keep4 = (comp[4][0][sel], comp[4][1][sel])
    # a compressed state holding only the selected entries, placed first, gives the same result
    # when the selection is "all of them"
    comp_sel = {4: keep4, 16: comp[16]}
    L_fake = L  # entries beyond len(sel) must not be read: pass sel = arange(len(sel))
    O2, _, _, _ = tree_verify_attn_request(cfg, parents, L_fake, Q, comp_sel, np.arange(len(sel)),
                                           rawK, rawV, treeK, treeV, g)
    np.testing.assert_allclose(O, O2, atol=1e-13)

"""Check (d): the state after refresh equals compressing prefix + accepted tokens from scratch."""

import json
import os

import numpy as np
import pytest

from oracle import compress_prefix, refresh_commit_request, verify_round, VerifyConfig
from oracle.storage import round_to_storage

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiny_tree.json")


@pytest.mark.parametrize("store", ["bf16", "f64"])
@pytest.mark.parametrize("L,path_len", [(250, 8), (253, 3), (255, 1), (127, 4), (120, 8)])
def test_refresh_equals_compress_from_scratch(store, L, path_len):
    rng = np.random.default_rng(L * 10 + path_len)
    d, D, ms = 16, 10, (4, 128)
    cap = L + D + 4
    rawK = np.zeros((cap, d))
    rawV = np.zeros((cap, d))
    rawK[:L] = round_to_storage(rng.standard_normal((L, d)), "bf16")
    rawV[:L] = round_to_storage(rng.standard_normal((L, d)), "bf16")
    treeK = round_to_storage(rng.standard_normal((D, d)), "bf16")
    treeV = round_to_storage(rng.standard_normal((D, d)), "bf16")
    g = {m: rng.standard_normal(d) for m in ms}
    comp = {}
    for m in ms:
        ck = np.full((cap // m + 1, d), 123.0)   # sentinel rows beyond the valid prefix
        cv = np.full((cap // m + 1, d), 123.0)
        ck[:L // m], cv[:L // m] = compress_prefix(rawK, rawV, L, m, g[m], store)
        comp[m] = (ck, cv)
    path = sorted(rng.choice(np.arange(1, D), size=path_len - 1, replace=False).tolist())
    path = [0] + path
    rK, rV = rawK.copy(), rawV.copy()
    L_new, committed = refresh_commit_request(ms, store, L, path, D, treeK, treeV, g, rK, rV, comp)
    assert L_new == L + path_len
    assert committed.tolist() == [L + i for i in range(path_len)] + [-1] * (D - path_len)
    # raw rows: the accepted tokens, bit for bit, rows before L untouched, rows after L_new untouched
    seqK = np.concatenate([rawK[:L], treeK[path]])
    seqV = np.concatenate([rawV[:L], treeV[path]])
    assert np.array_equal(rK[:L_new], seqK)
    assert np.array_equal(rV[:L_new], seqV)
    assert np.array_equal(rK[L_new:], rawK[L_new:])
    for m in ms:
        CK, CV = compress_prefix(seqK, seqV, L_new, m, g[m], store)
        assert np.array_equal(comp[m][0][:L_new // m], CK)
        assert np.array_equal(comp[m][1][:L_new // m], CV)
        assert np.all(comp[m][0][L_new // m:] == 123.0)


def test_capacity_is_enforced():
    d = 4
    raw = np.zeros((10, d))
    comp = {4: (np.zeros((3, d)), np.zeros((3, d)))}
    with pytest.raises(ValueError):
        refresh_commit_request((4,), "f64", 8, [0, 1, 2], 3, np.ones((3, d)), np.ones((3, d)),
                               {4: np.zeros(d)}, raw, raw.copy(), comp)


def test_commit_fills_every_capacity_exactly():
    # raw rows and compressed entries end exactly at their capacities: the last committed token
    # closes the last block that fits, and the commit succeeds
    rng = np.random.default_rng(5)
    d, D, m, L = 8, 4, 4, 8
    raw = np.zeros((L + D, d))
    rawV = np.zeros((L + D, d))
    raw[:L] = rng.standard_normal((L, d))
    rawV[:L] = rng.standard_normal((L, d))
    treeK = rng.standard_normal((D, d))
    treeV = rng.standard_normal((D, d))
    g = {m: rng.standard_normal(d)}
    ck, cv = np.zeros(((L + D) // m, d)), np.zeros(((L + D) // m, d))
    ck[:L // m], cv[:L // m] = compress_prefix(raw, rawV, L, m, g[m], "f64")
    comp = {m: (ck, cv)}
    L_new, _ = refresh_commit_request((m,), "f64", L, [0, 1, 2, 3], D, treeK, treeV, g, raw, rawV,
                                      comp)
    assert L_new == L + D == raw.shape[0]
    CK, CV = compress_prefix(raw, rawV, L_new, m, g[m], "f64")
    assert np.array_equal(ck, CK) and np.array_equal(cv, CV)


def test_tiny_round_golden():
    from tree_speculative_verify_gb300 import workloads
    with open(GOLDEN) as f:
        gold = json.load(f)
    wl = workloads.tiny()
    cfg = VerifyConfig(H=wl.H, d=wl.d, ms=wl.ms, W=wl.W, tail_mode=wl.tail_mode, store="f32")
    rawK = wl.rawK.numpy()
    rawV = wl.rawV.numpy()
    g = {m: wl.g[m].numpy() for m in wl.ms}
    comp = {}
    for m in wl.ms:
        ck = np.zeros((1, wl.cap4, wl.d))
        cv = np.zeros((1, wl.cap4, wl.d))
        ck[0, :wl.L[0] // m], cv[0, :wl.L[0] // m] = compress_prefix(rawK[0], rawV[0], int(wl.L[0]), m, g[m], "f32")
        comp[m] = (ck, cv)
    res = verify_round(cfg, wl.parents, wl.L, wl.Q.numpy(), comp, None, rawK, rawV,
                       wl.treeK.numpy(), wl.treeV.numpy(), g, wl.draft, wl.target)[0]
    assert res["path"] == gold["accept_path"]
    assert res["accept_len"] == gold["accept_len"]
    assert res["L_new"] == gold["L_after_commit"]
    assert res["committed"].tolist() == gold["committed_pos"]
    assert res["scratch"] == {}          # L = 256 and depth <= 2: no node closes a 4-block
    assert res["entries"] == {}


@pytest.mark.parametrize("L", [250, 253])
def test_round_reports_the_rows_and_entries_it_commits(L):
    # a 2-request round over two different branching trees: what the round reports as written
    # (raw rows, compressed entries, new length) equals rebuilding prefix + accepted path from
    # scratch, each request with its own tree and tokens
    rng = np.random.default_rng(L)
    B, D, d, H, W, ms = 2, 7, 8, 2, 6, (4, 128)
    parents = np.array([[-1, 0, 0, 1, 1, 3, 4], [-1, 0, 1, 1, 2, 0, 5]])
    cap = L + D + 4
    rawK = np.zeros((B, cap, d))
    rawV = np.zeros((B, cap, d))
    rawK[:, :L] = rng.standard_normal((B, L, d))
    rawV[:, :L] = rng.standard_normal((B, L, d))
    treeK = rng.standard_normal((B, D, d))
    treeV = rng.standard_normal((B, D, d))
    Q = rng.standard_normal((B, D, H, d))
    g = {m: rng.standard_normal(d) for m in ms}
    comp = {}
    for m in ms:
        ck = np.zeros((B, cap // m + 1, d))
        cv = np.zeros((B, cap // m + 1, d))
        for b in range(B):
            ck[b, :L // m], cv[b, :L // m] = compress_prefix(rawK[b], rawV[b], L, m, g[m], "f64")
        comp[m] = (ck, cv)
    draft = np.array([[9, 1, 2, 3, 4, 5, 6]] * B)
    # request 0 accepts 0 -> 1 -> 3 -> 5 (bonus 40); request 1 accepts 0 -> 5 -> 6 (bonus 42)
    target = np.array([[1, 3, 41, 5, 0, 40, 0], [5, 0, 0, 0, 0, 6, 42]])
    cfg = VerifyConfig(H=H, d=d, ms=ms, W=W, tail_mode="window", store="f64")
    res = verify_round(cfg, parents, np.array([L, L]), Q, comp, None, rawK, rawV, treeK, treeV, g,
                       draft, target)
    for b, (path, bonus) in enumerate([([0, 1, 3, 5], 40), ([0, 5, 6], 42)]):
        r = res[b]
        assert r["path"] == path and r["accept_len"] == len(path) and r["bonus"] == bonus
        assert r["L_new"] == L + len(path)
        seqK = np.concatenate([rawK[b, :L], treeK[b, path]])
        seqV = np.concatenate([rawV[b, :L], treeV[b, path]])
        assert np.array_equal(r["raw_rows"][0], treeK[b, path])
        assert np.array_equal(r["raw_rows"][1], treeV[b, path])
        want = {(m, (e + 1) // m - 1) for m in ms for e in range(L, L + len(path)) if (e + 1) % m == 0}
        assert set(r["entries"]) == want
        for (m, j), (ck, cv) in r["entries"].items():
            CK, CV = compress_prefix(seqK, seqV, L + len(path), m, g[m], "f64")
            assert np.array_equal(ck, CK[j]) and np.array_equal(cv, CV[j])


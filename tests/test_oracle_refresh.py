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

"""The bench's algorithmic accounting agrees with the visible sets the oracle builds.

``bench.py`` reports the attention's achieved TFLOP/s and GB/s from its own bookkeeping of how
many entries every tree node attends to (``visible_counts``: the compressed prefix or the
selection, the C128 entries, the raw window, the node's ancestors inside the window and the
scratch entries of its block-closing ancestors) and of the rows one request reads.  Here the
same workloads go through the oracle's ``visible_set``: every node's count must equal the number
of rows the oracle attends over, the tail rows must be the union of the nodes' raw windows, and
the scratch rows the number of entries the scratch pad holds.
"""

import numpy as np
import pytest

import bench
import oracle
from tree_speculative_verify_gb300 import workloads


def _cases():
    return {
        "window_ragged": lambda: workloads.make_workload(
            "acct_window", B=3, D=8, H=2, d=8, W=128, tail_mode="window", ms=(4, 128),
            dtype="bf16", L=[1021, 100, 255], k=2, steps=4, p_match=0.55, seed=31, kv_scale=0.5),
        "remainder": lambda: workloads.make_workload(
            "acct_rem", B=2, D=6, H=2, d=8, W=0, tail_mode="remainder", ms=(4,), dtype="f32",
            L=[253, 64], k=2, steps=3, p_match=0.6, seed=32, kv_scale=1.0),
        "c128_only": lambda: workloads.make_workload(
            "acct_c128", B=2, D=8, H=2, d=8, W=16, tail_mode="window", ms=(128,), dtype="bf16",
            L=[383, 129], k=2, steps=4, p_match=0.55, seed=33, kv_scale=0.5),
        "chain_24": lambda: workloads.make_workload(
            "acct_chain", B=2, D=24, H=2, d=8, W=8, tail_mode="window", ms=(4, 128), dtype="bf16",
            L=[250, 7], k=1, steps=23, p_match=0.6, seed=34, kv_scale=0.5),
        "selection": lambda: workloads.long_context(B=2, L=(2000, 3000), n_sel=64),
    }


@pytest.mark.parametrize("case", list(_cases()))
def test_visible_counts_equal_the_oracle_visible_sets(case):
    wl = _cases()[case]()
    counts = bench.visible_counts(wl)
    cfg = oracle.VerifyConfig(H=wl.H, d=wl.d, ms=tuple(wl.ms), W=wl.W, tail_mode=wl.tail_mode,
                              store="f64")
    d = wl.d
    for b in range(wl.B):
        L = int(wl.L[b])
        par = [int(x) for x in wl.parents[b]]
        plan = oracle.build_plan(par, L, wl.W, wl.tail_mode, tuple(wl.ms))
        # the count of rows does not depend on their values: zero arrays of the right sizes
        raw = np.zeros((L + wl.D + 1, d))
        tree = np.zeros((wl.D, d))
        comp = {m: (np.zeros((L // m + 1, d)), np.zeros((L // m + 1, d))) for m in wl.ms}
        g = {m: np.zeros(d) for m in wl.ms}
        scratch = oracle.scratch_entries(cfg, par, L, raw, raw, tree, tree, g, plan)
        sel = None if not wl.n_sel else wl.sel[b]
        raw_rows = set()
        for v in range(wl.D):
            K, _ = oracle.visible_set(cfg, v, plan, L, comp, sel, raw, raw, tree, tree, scratch)
            assert K.shape[0] == counts[b]["per_node"][v], f"request {b}, node {v}"
            raw_rows |= set(range(plan.raw_lo[v], L))
        assert counts[b]["tail"] == len(raw_rows)
        assert counts[b]["scr"] == len(scratch)
        assert counts[b]["tree"] == wl.D
        n_shared = (len(sel) if sel is not None else L // 4) if 4 in wl.ms else 0
        n_shared += L // 128 if 128 in wl.ms else 0
        assert counts[b]["shared"] == n_shared


def test_flops_and_bytes_follow_the_counts():
    wl = _cases()["window_ragged"]()
    counts = bench.visible_counts(wl)
    kv_bytes, qo_bytes, flops = bench.attention_accounting(wl)
    es = 2
    # 2 flops per multiply-add, for Q.K and for P.V, per head and visible entry
    assert flops == sum(2 * 2 * wl.d * wl.H * n for c in counts for n in c["per_node"])
    assert kv_bytes == sum((c["shared"] + c["tail"] + c["tree"] + c["scr"]) * 2 * wl.d * es
                           for c in counts)
    assert qo_bytes == 2 * wl.B * wl.D * wl.H * wl.d * es

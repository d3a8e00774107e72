"""GPU parity: the CUDA path against the oracle on the same seeded inputs (one full round).

Integers (ancestor masks, depths, window bounds, scratch visibility, accept lengths, paths,
bonus tokens, committed positions, new lengths, committed raw rows) must match bit for bit;
floats within the tolerances of tests/helpers.py.
"""

import numpy as np
import pytest
import torch

from tree_speculative_verify_gb300 import _lib, workloads
from helpers import check_round, gpu_round, oracle_prefix, run_oracle

pytestmark = pytest.mark.gpu

KERNELS = {"auto": _lib.TV_ATTN_AUTO, "simt": _lib.TV_ATTN_SIMT}


def _run(wl, kernel="auto", requests=None):
    comp = oracle_prefix(wl)
    reqs = list(range(wl.B)) if requests is None else requests
    res = run_oracle(wl, comp, requests=reqs)
    shape, st0, st, rb = gpu_round(wl, KERNELS[kernel], comp=comp)
    return check_round(wl, res, st0, st, rb, reqs)


@pytest.mark.parametrize("L", [256, 253, 254, 255])
def test_tiny_fp32(L):
    _run(workloads.tiny(L=L))


@pytest.mark.parametrize("kernel", ["auto", "simt"])
def test_small_bf16_full_size(kernel):
    _run(workloads.small(), kernel)


@pytest.mark.parametrize("kernel", ["auto", "simt"])
def test_serving_reduced_batch(kernel):
    # several KV tiles per request, ragged tails, scratch entries of both compressors
    wl = workloads.make_workload("serving_small", B=6, D=8, H=64, d=512, W=128,
                                 tail_mode="window", ms=(4, 128), dtype="bf16", L=(1021, 2300),
                                 k=2, steps=4, p_match=0.55, seed=3, kv_scale=0.5)
    _run(wl, kernel)


def test_serving_full_size_sampled():
    wl = workloads.serving()
    longest = int(np.argmax(wl.L))
    _run(wl, "auto", requests=sorted({0, 17, 42, 63, longest}))


@pytest.mark.parametrize("kernel", ["auto", "simt"])
def test_long_context_reduced(kernel):
    wl = workloads.long_context(B=2, L=(9000, 12000), n_sel=512)
    _run(wl, kernel)


def test_long_context_full_size_sampled():
    wl = workloads.long_context()
    _run(wl, "auto", requests=[0, int(np.argmax(wl.L))])


@pytest.mark.parametrize("idx", [0, 9, 26, 37, 52, 63])
def test_sweep_cells(idx):
    cell = workloads.sweep_cells()[idx]
    B = min(cell["B"], 4)
    wl = workloads.sweep_cell(idx, cell["D"], B, cell["kind"], cell["p"])
    _run(wl)


def _serving_like(name, B, L, seed):
    return workloads.make_workload(name, B=B, D=8, H=64, d=512, W=128, tail_mode="window",
                                   ms=(4, 128), dtype="bf16", L=L, k=2, steps=4, p_match=0.55,
                                   seed=seed, kv_scale=0.5)


def test_more_work_items_than_cta_pairs():
    # 48 requests x 2 row-tile pairs x 2 value halves = 192 work items of ragged sizes: more than
    # the CTA pairs that fit on the device at once, so later items start as earlier ones finish
    _run(_serving_like("many_items", 48, (200, 900), 22))


def test_split_kv_with_empty_chunks():
    # 12 requests up to 8191 tokens: the KV tiles are split into chunks (fp32 partials + merge),
    # 144 work items; the nearly empty requests (L = 0, 1, 3) leave later chunks without a tile
    Ls = [8000, 0, 7000, 3, 8100, 64, 7900, 129, 6000, 1, 8191, 500]
    _run(_serving_like("split_items", 12, Ls, 21))


# --- edge cases ------------------------------------------------------------------------------

def _edge(name, **kw):
    base = dict(B=3, D=8, H=16, d=512, W=128, tail_mode="window", ms=(4, 128), dtype="bf16",
                L=300, k=2, steps=4, p_match=0.6, seed=11, kv_scale=0.5)
    base.update(kw)
    return workloads.make_workload(name, **base)


@pytest.mark.parametrize("L", [0, 1, 3, 5, 127, 128, 131, 255])
def test_short_prefixes(L):
    # empty prefix, prefixes shorter than the window and than one C128 block, roots that close
    # a C128 block (L = 127, 255) and nodes that close one
    _run(_edge(f"short{L}", L=L, seed=L))


def test_root_only_tree():
    _run(_edge("root_only", D=1, k=1, steps=0))


def test_max_budget_tree():
    # D = 64 nodes: two 32-lane halves in the walk and 64-bit masks fully used
    _run(_edge("d64", D=64, k=2, steps=6, H=2, L=(500, 700), B=2))


def test_long_chain_crosses_c4_blocks():
    _run(_edge("chain24", D=24, k=1, steps=23, H=4, L=(120, 140), B=4))


def test_small_head_dim_fp32_window():
    _run(_edge("f32_d64", d=64, H=8, dtype="f32", L=(40, 300), B=5))


def test_bf16_head_dim_128():
    _run(_edge("bf16_d128", d=128, H=32, L=(129, 1000), B=4))


def test_c128_only_and_c4_only():
    _run(_edge("c128only", ms=(128,), L=(300, 700)))
    _run(_edge("c4only", ms=(4,), L=(300, 700)))


def test_remainder_tail_bf16():
    _run(_edge("remainder", tail_mode="remainder", W=0, ms=(4,), L=(97, 203), B=4))


def test_tiny_window():
    _run(_edge("w3", W=3, L=(10, 90), B=4, D=10, k=2, steps=4))


def test_two_rounds_in_a_row():
    """The state committed by one round is the state the next round verifies against."""
    wl = _edge("tworounds", L=(250, 400), B=4, D=8)
    comp = oracle_prefix(wl)
    res = run_oracle(wl, comp)
    shape, st0, st, rb = gpu_round(wl, comp=comp)
    check_round(wl, res, st0, st, rb, range(wl.B))
    # second round: new tree inputs, same committed state as the oracle's
    wl2 = _edge("tworounds2", L=(250, 400), B=4, D=8, seed=99)
    wl2.L = np.array([res[b]["L_new"] for b in range(wl.B)])
    # the oracle's own committed raw rows on top of the first workload's prefix
    wl2.rawK = wl.rawK.clone()
    wl2.rawV = wl.rawV.clone()
    for b in range(wl.B):
        L0, L1 = int(wl.L[b]), res[b]["L_new"]
        wl2.rawK[b, L0:L1] = torch.from_numpy(res[b]["raw_rows"][0]).to(wl.rawK.dtype)
        wl2.rawV[b, L0:L1] = torch.from_numpy(res[b]["raw_rows"][1]).to(wl.rawV.dtype)
    # the oracle state for the second verify round: its own committed entries on top of its prefix
    comp2 = {m: (comp[m][0].copy(), comp[m][1].copy()) for m in comp}
    for b in range(wl.B):
        for (m, j), (ck, cv) in res[b]["entries"].items():
            comp2[m][0][b, j] = ck
            comp2[m][1][b, j] = cv
    # raw rows committed by the first verify round are bit-equal on both sides (checked above)
    res2 = run_oracle(wl2, comp2)
    from tree_speculative_verify_gb300 import engine
    rb2 = engine.alloc_round(wl2, shape)
    st_before = st.clone()
    engine.verify_round(shape, st, rb2)
    torch.cuda.synchronize()
    check_round(wl2, res2, st_before, st, rb2, range(wl.B))


@pytest.mark.parametrize("name", ["tiny", "small", "serving_reduced", "c128_boundary"])
def test_prefill_compress_matches_oracle(name):
    """tv_prefill_compress writes every complete C4 / C128 block of the committed prefix."""
    from helpers import TOL, close, np32
    if name == "tiny":
        wl = workloads.tiny(L=255)
    elif name == "small":
        wl = workloads.small()
    elif name == "serving_reduced":
        wl = workloads.serving(B=5, L=(1000, 3000))
    else:
        wl = _edge("c128b", L=(255, 640), B=4)
    from tree_speculative_verify_gb300 import engine
    shape = engine.shape_for(wl)
    st = engine.alloc_state(wl)
    rb = engine.alloc_round(wl, shape)
    engine.prefill(shape, st, rb)
    torch.cuda.synchronize()
    assert int(rb.status.item()) == 0
    comp = oracle_prefix(wl)
    tol = TOL[wl.dtype]
    for m in wl.ms:
        gk = np32(st.c4K if m == 4 else st.c128K)
        gv = np32(st.c4V if m == 4 else st.c128V)
        for b in range(wl.B):
            n = int(wl.L[b]) // m
            close(gk[b, :n], comp[m][0][b, :n], tol, f"prefill C{m} K request {b}")
            close(gv[b, :n], comp[m][1][b, :n], tol, f"prefill C{m} V request {b}")
            assert np.all(gk[b, n:] == 0)      # nothing written beyond the valid entries

"""GPU indexer top-k (tv_indexer_topk) against the oracle: the selection lists must be identical
(integers, bit-exact); the scores are fixed to one fp32 summation order on both sides."""

import numpy as np
import pytest
import torch

import oracle
from tree_speculative_verify_gb300 import _lib, engine, workloads
from helpers import check_round, gpu_round, oracle_prefix, run_oracle

pytestmark = pytest.mark.gpu


def _gpu_select(wl, L=None, n_sel=None):
    shape = engine.shape_for(wl)
    if n_sel is not None:
        shape.n_sel = n_sel
    q = wl.q_idx.cuda()
    k = wl.k_idx.cuda()
    Lt = torch.as_tensor(wl.L if L is None else L, dtype=torch.int32).cuda()
    sel = torch.full((wl.B, shape.n_sel), -5, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(_lib.tv_indexer_workspace_size(shape), 256), dtype=torch.uint8,
                     device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _lib.tv_indexer_topk(shape, 64, q, k, Lt, sel, ws, status)
    torch.cuda.synchronize()
    return sel.cpu().numpy(), int(status.item())


def _oracle_select(wl, b, n_sel=None):
    return oracle.indexer_select(wl.q_idx[b].float().numpy(), wl.k_idx[b].float().numpy(),
                                 int(wl.L[b]), wl.n_sel if n_sel is None else n_sel)


@pytest.mark.parametrize("B,L,n_sel", [(3, (3000, 9000), 256), (4, (1030, 1100), 257),
                                        (2, (8192, 8192), 2048)])
def test_selection_matches_oracle(B, L, n_sel):
    wl = workloads.long_context(B=B, L=L, n_sel=n_sel)
    got, status = _gpu_select(wl)
    assert status == 0
    for b in range(B):
        assert np.array_equal(got[b], _oracle_select(wl, b)), f"request {b}"


def test_full_size_selection_matches_oracle():
    wl = workloads.long_context()
    got, status = _gpu_select(wl)
    assert status == 0
    for b in range(wl.B):
        assert np.array_equal(got[b], _oracle_select(wl, b)), f"request {b}"


def test_exact_ties_go_to_the_lower_index():
    wl = workloads.long_context(B=2, L=(2000, 2100), n_sel=100)
    # integer-valued keys with many duplicates: exact ties at the selection boundary
    rng = np.random.default_rng(7)
    wl.q_idx = torch.from_numpy(rng.integers(-2, 3, size=(2, 64)).astype(np.float32)).bfloat16()
    k = rng.integers(-1, 2, size=(2, wl.cap4, 64)).astype(np.float32)
    k[:, 50:400] = k[:, 10:11]            # 350 copies of one key
    wl.k_idx = torch.from_numpy(k).bfloat16()
    got, status = _gpu_select(wl)
    assert status == 0
    for b in range(2):
        want = _oracle_select(wl, b)
        assert np.array_equal(got[b], want), f"request {b}"


def test_more_entries_than_shared_memory_holds():
    # 42500 C4 entries: above the 40960 keys the select kernel stages, so every pass re-reads the
    # scores from global memory
    wl = workloads.long_context(B=1, L=(170000, 170000), n_sel=2048)
    got, status = _gpu_select(wl)
    assert status == 0
    assert np.array_equal(got[0], _oracle_select(wl, 0))


def test_all_scores_equal():
    # a zero query: every score is 0, all keys tie, the lowest n_sel indices are kept
    wl = workloads.long_context(B=2, L=(3000, 5000), n_sel=300)
    wl.q_idx = torch.zeros_like(wl.q_idx)
    got, status = _gpu_select(wl)
    assert status == 0
    for b in range(2):
        want = _oracle_select(wl, b)
        assert np.array_equal(want, np.arange(300))
        assert np.array_equal(got[b], want), f"request {b}"


def test_too_few_entries_is_reported_per_request():
    wl = workloads.long_context(B=3, L=(3000, 3100), n_sel=64)
    L = wl.L.copy()
    L[1] = 4 * 63 + 3                    # 63 C4 entries < n_sel
    got, status = _gpu_select(wl, L=L)
    assert status == -9
    assert np.all(got[1] == -1)
    for b in (0, 2):
        assert np.array_equal(got[b], oracle.indexer_select(
            wl.q_idx[b].float().numpy(), wl.k_idx[b].float().numpy(), int(L[b]), 64))


def test_indexer_feeds_the_tensor_core_attention():
    # the round's sparse path end to end: device selection -> tree-verify attention, against the
    # oracle round run on the oracle's own selection
    wl = workloads.long_context(B=2, L=(9000, 12000), n_sel=512)
    sel_gpu, status = _gpu_select(wl)
    assert status == 0
    wl.sel = np.stack([_oracle_select(wl, b) for b in range(wl.B)])
    assert np.array_equal(sel_gpu, wl.sel)
    comp = oracle_prefix(wl)
    res = run_oracle(wl, comp)
    shape, st0, st, rb = gpu_round(wl, comp=comp)
    check_round(wl, res, st0, st, rb, range(wl.B))

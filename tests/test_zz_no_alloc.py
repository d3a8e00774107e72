"""The allocation-free attention entry point matches the workspace one.

tv_tree_verify_attn_noalloc serves callers that cannot allocate device memory (an engine whose page
pool owns all free memory, a decode loop that cannot afford cudaMalloc's implicit synchronisation,
a plug-in host without an allocator): it keeps the split-KV partials in the library's built-in
scratch array instead of a caller workspace.  This file is collected last so that a failure here
never hides another test's result.
"""

import math

import numpy as np
import pytest
import torch

from tree_speculative_verify_gb300 import _lib, engine, workloads
from helpers import TOL, np32

pytestmark = pytest.mark.gpu


def _prepared(wl, kernel=_lib.TV_ATTN_AUTO):
    shape = engine.shape_for(wl, kernel)
    st = engine.alloc_state(wl)
    rb = engine.alloc_round(wl, shape)
    engine.prefill(shape, st, rb)
    engine.plan(shape, st, rb)
    engine.branch_compress(shape, st, rb)
    torch.cuda.synchronize()
    assert int(rb.status.item()) == 0
    return shape, st, rb


def _noalloc(shape, st, rb, O, lse):
    _lib.tv_tree_verify_attn_noalloc(
        shape, rb.Q, st.c4K, st.c4V, rb.sel, st.c128K, st.c128V, st.rawK, st.rawV, st.L, rb.treeK,
        rb.treeV, rb.anc, rb.raw_lo, rb.vis4, rb.vis128, rb.scrK4, rb.scrV4, rb.scrK128,
        rb.scrV128, 1.0 / math.sqrt(shape.d), O, lse, rb.status)


@pytest.mark.parametrize("case", ["small_split_kv", "tiny_fp32", "selection_list"])
def test_noalloc_matches_workspace_entry_point_twice(case):
    if case == "small_split_kv":
        # 4 requests: the attention splits every request's KV over many CTAs, so the partials
        # fill most of the built-in scratch
        wl = workloads.small()
    elif case == "selection_list":
        # the tensor-core path gathers the selected C4 rows into the scratch first
        wl = workloads.long_context(B=2, L=(9000, 12000), n_sel=512)
    else:
        wl = workloads.tiny(L=255)
    shape, st, rb = _prepared(wl)
    assert _lib.tv_workspace_size(shape) > 256   # the scratch path is really exercised
    engine.attention(shape, st, rb)
    torch.cuda.synchronize()
    ref_O, ref_lse = np32(rb.O), rb.lse.cpu().numpy()
    tol = TOL[wl.dtype]
    for _ in range(2):
        O = torch.full_like(rb.O, float("nan"))
        lse = torch.full_like(rb.lse, float("nan"))
        _noalloc(shape, st, rb, O, lse)
        torch.cuda.synchronize()
        assert int(rb.status.item()) == 0
        got = np32(O)
        err = np.abs(got - ref_O)
        assert np.all(np.isfinite(got))
        assert err.max() <= tol["max_abs"] and err.mean() <= tol["mean_abs"]
        assert np.abs(lse.cpu().numpy() - ref_lse).max() <= tol["lse"]


def test_noalloc_rejects_shapes_beyond_its_scratch():
    wl = workloads.long_context(B=2, L=(3000, 3100), n_sel=64)
    shape = engine.shape_for(wl)
    shape.B = 4096                     # far more split-KV partials than the built-in scratch holds
    shape.c4_cap = 20000
    need = _lib.tv_workspace_size(shape)
    assert need > (32 << 20)
    with pytest.raises(_lib.TreeVerifyError) as e:
        dummy = torch.zeros(1, device="cuda")
        _lib.tv_tree_verify_attn_noalloc(shape, *([dummy] * 19), 0.05, dummy, dummy,
                                         torch.zeros(1, dtype=torch.int32, device="cuda"))
    assert e.value.code == -7


def test_prepare_then_calls_take_no_device_memory():
    """After tv_noalloc_prepare, the entry point takes no device memory: the free memory the
    driver reports is the same before and after several calls."""
    _lib.tv_noalloc_prepare()
    wl = workloads.small()
    shape, st, rb = _prepared(wl)
    O = torch.empty_like(rb.O)
    lse = torch.empty_like(rb.lse)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        _noalloc(shape, st, rb, O, lse)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert int(rb.status.item()) == 0
    assert free1 == free0, (free0, free1)


def test_host_errors_name_the_noalloc_entry_point():
    wl = workloads.small()
    shape, st, rb = _prepared(wl)
    with pytest.raises(_lib.TreeVerifyError) as e:
        _lib.tv_tree_verify_attn_noalloc(
            shape, rb.Q, st.c4K, st.c4V, rb.sel, st.c128K, st.c128V, st.rawK, st.rawV, st.L,
            rb.treeK, rb.treeV, rb.anc, rb.raw_lo, rb.vis4, rb.vis128, rb.scrK4, rb.scrV4,
            rb.scrK128, rb.scrV128, -1.0, rb.O, rb.lse, rb.status)
    # the library's own message (not the binding's prefix) names the entry point
    assert _lib.load().tv_last_error_string().decode().startswith("tv_tree_verify_attn_noalloc")

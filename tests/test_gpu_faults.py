"""Device-side error reporting: malformed inputs set the caller's status word (first error wins),
the other requests' results stay valid, and the context stays usable.  Faults are injected on the
host (corrupted inputs); nothing here traps or hangs the GPU."""

import numpy as np
import pytest
import torch

from tree_speculative_verify_gb300 import _lib, engine, workloads
from helpers import check_round, oracle_prefix, run_oracle

pytestmark = pytest.mark.gpu


def _wl(**kw):
    base = dict(B=3, D=6, H=16, d=512, W=128, tail_mode="window", ms=(4, 128), dtype="bf16",
                L=300, k=2, steps=3, p_match=0.6, seed=21, kv_scale=0.5)
    base.update(kw)
    return workloads.make_workload("faults", **base)


def _setup(wl):
    shape = engine.shape_for(wl)
    st = engine.alloc_state(wl)
    rb = engine.alloc_round(wl, shape)
    return shape, st, rb


def test_bad_tree_sets_status_and_leaves_other_requests_valid():
    wl = _wl()
    comp = oracle_prefix(wl)
    res = run_oracle(wl, comp, requests=[0, 2], with_refresh=False)
    shape, st, rb = _setup(wl)
    from helpers import upload_prefix
    upload_prefix(wl, st, comp)
    bad = rb.parents.clone()
    bad[1, 3] = 5                      # a parent numbered after its child
    rb.parents.copy_(bad)
    engine.plan(shape, st, rb)
    engine.branch_compress(shape, st, rb)
    engine.attention(shape, st, rb)
    engine.accept(shape, st, rb)
    torch.cuda.synchronize()
    assert int(rb.status.item()) == -3
    # request 1's plan is zeroed, requests 0 and 2 match the oracle
    assert torch.all(rb.anc[1] == 0)
    O = rb.O.float().cpu().numpy()
    for b in (0, 2):
        err = np.abs(O[b] - res[b]["O"])
        assert err.max() <= 2e-2 and err.mean() <= 2e-3
        assert int(rb.accept_len[b].item()) == res[b]["accept_len"]
    # the context is still usable
    rb.status.zero_()
    rb.parents.copy_(torch.as_tensor(wl.parents, dtype=torch.int32))
    engine.plan(shape, st, rb)
    torch.cuda.synchronize()
    assert int(rb.status.item()) == 0


def test_capacity_overflow_in_refresh_is_reported_and_request_untouched():
    wl = _wl(L=(290, 300))
    shape, st, rb = _setup(wl)
    engine.prefill(shape, st, rb)
    engine.verify_round(shape, st, rb, commit=False)
    torch.cuda.synchronize()
    assert int(rb.status.item()) == 0
    # force request 0 to the end of its raw capacity: committing n >= 1 rows must overflow
    L_full = torch.tensor([wl.raw_cap], dtype=torch.int32, device="cuda")
    st.L[0:1].copy_(L_full)
    raw_before = st.rawK[0].clone()
    L_before = st.L.clone()
    engine.refresh(shape, st, rb)
    torch.cuda.synchronize()
    assert int(rb.status.item()) == -4
    assert int(st.L[0].item()) == wl.raw_cap
    assert torch.equal(st.rawK[0], raw_before)
    assert torch.all(rb.committed[0] == -1)
    # the other requests committed normally
    n = rb.accept_len.cpu()
    for b in (1, 2):
        assert int(st.L[b].item()) == int(L_before[b].item()) + int(n[b])


def test_selection_index_out_of_range_is_reported():
    wl = workloads.long_context(B=2, L=(3000, 3100), n_sel=64)
    wl.sel = wl.sel.copy()
    wl.sel[1, 5] = int(wl.L[1]) // 4 + 10       # beyond the request's C4 entries
    shape, st, rb = _setup(wl)
    engine.prefill(shape, st, rb)
    engine.verify_round(shape, st, rb, commit=False)
    torch.cuda.synchronize()
    assert int(rb.status.item()) == -9
    assert torch.isfinite(rb.O.float()).all()


def test_host_validation_rejects_null_before_launch():
    wl = _wl()
    shape, st, rb = _setup(wl)
    with pytest.raises(_lib.TreeVerifyError) as e:
        _lib.tv_accept_walk(shape, rb.parents, None, rb.target, rb.accept_len, rb.path, rb.bonus,
                            rb.status)
    assert e.value.code == -1
    with pytest.raises(_lib.TreeVerifyError) as e:
        small_ws = torch.empty(256, dtype=torch.uint8, device="cuda")
        big = engine.shape_for(wl, _lib.TV_ATTN_SIMT)
        _lib.tv_tree_verify_attn(big, rb.Q, st.c4K, st.c4V, None, st.c128K, st.c128V, st.rawK,
                                 st.rawV, st.L, rb.treeK, rb.treeV, rb.anc, rb.raw_lo, rb.vis4,
                                 rb.vis128, rb.scrK4, rb.scrV4, rb.scrK128, rb.scrV128, 0.04, rb.O,
                                 rb.lse, small_ws, rb.status)
    assert e.value.code == -7


def test_attention_wait_that_runs_out_reports_timeout_and_context_stays_usable():
    """A bounded device-side wait runs out on purpose: with tv_debug_attn_timeout the tensor-core
    attention's producers never issue the K copies of KV tile 2, so the MMA issuer's wait for that
    tile expires after 200 us.  The kernel records TV_ERR_TIMEOUT, stops both CTAs of the pair,
    drains the copies and MMAs it did issue and returns; nothing traps or hangs.  The next call on
    the same context matches the oracle."""
    from helpers import upload_prefix
    wl = _wl(B=2, L=(700, 900))       # 5 KV tiles per request: C4 x2, C128, raw tail, extra
    comp = oracle_prefix(wl)
    res = run_oracle(wl, comp, with_refresh=False)
    shape, st, rb = _setup(wl)
    assert _lib.tv_attn_kernel_for(shape) == _lib.TV_ATTN_TCGEN05
    upload_prefix(wl, st, comp)
    engine.plan(shape, st, rb)
    engine.branch_compress(shape, st, rb)
    torch.cuda.synchronize()
    assert int(rb.status.item()) == 0
    _lib.tv_debug_attn_timeout(200_000, 2)
    try:
        engine.attention(shape, st, rb)
        torch.cuda.synchronize()
    finally:
        _lib.tv_debug_attn_timeout(2_000_000_000, -1)
    assert int(rb.status.item()) == -8
    # the context is still usable and the next call is exact again
    rb.status.zero_()
    rb.O.fill_(float("nan"))
    engine.attention(shape, st, rb)
    torch.cuda.synchronize()
    assert int(rb.status.item()) == 0
    O = rb.O.float().cpu().numpy()
    lse = rb.lse.cpu().numpy()
    for b in range(wl.B):
        err = np.abs(O[b] - res[b]["O"])
        assert err.max() <= 2e-2 and err.mean() <= 2e-3
        assert np.abs(lse[b] - res[b]["LSE"]).max() <= 1e-2

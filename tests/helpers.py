"""Shared test plumbing: oracle-side state from a workload, GPU round runner, comparisons.

Tolerances (the float bar of the parity tests):
* bf16 caches, fp32 accumulation: O max-abs <= 2e-2 and mean-abs <= 2e-3; compressed entries
  (scratch pad and committed) the same; LSE max-abs <= 1e-2 (the tensor-core kernel multiplies
  V by probabilities rounded to bf16, a relative error of at most 2^-9 per term, so the row sums
  that set LSE agree to ~1e-3 of their value);
* fp32 caches: O and compressed entries max-abs <= 1e-4, LSE max-abs <= 1e-4.
"""

import math

import numpy as np
import torch

import oracle
from tree_speculative_verify_gb300 import engine, _lib

TOL = {
    "bf16": dict(max_abs=2e-2, mean_abs=2e-3, lse=1e-2),
    "f32": dict(max_abs=1e-4, mean_abs=1e-4, lse=1e-4),
}


def np32(t):
    """Stored tensor (fp32 or bf16, any device) -> exact float32 numpy array."""
    return t.detach().to("cpu").float().numpy()


def oracle_cfg(wl):
    return oracle.VerifyConfig(H=wl.H, d=wl.d, ms=wl.ms, W=wl.W, tail_mode=wl.tail_mode,
                               store=wl.dtype)


def oracle_prefix(wl):
    """Persistent compressed entries of every request, made by the oracle and rounded to the
    storage dtype: {m: (CK [B, cap_m, d], CV)} as float32 arrays (bf16 values are exact)."""
    out = {}
    for m in wl.ms:
        cap = wl.cap4 if m == 4 else wl.cap128
        CK = np.zeros((wl.B, cap, wl.d), dtype=np.float32)
        CV = np.zeros((wl.B, cap, wl.d), dtype=np.float32)
        for b in range(wl.B):
            L = int(wl.L[b])
            rk = np32(wl.rawK[b, :L])
            rv = np32(wl.rawV[b, :L])
            ck, cv = oracle.compress_prefix(rk, rv, L, m, np32(wl.g[m]), wl.dtype)
            CK[b, :L // m] = ck
            CV[b, :L // m] = cv
        out[m] = (CK, CV)
    return out


def upload_prefix(wl, st, comp):
    for m, (CK, CV) in comp.items():
        dstK, dstV = (st.c4K, st.c4V) if m == 4 else (st.c128K, st.c128V)
        dstK.copy_(torch.from_numpy(CK).to(dstK.dtype))
        dstV.copy_(torch.from_numpy(CV).to(dstV.dtype))


def run_oracle(wl, comp, requests=None, with_refresh=True):
    g = {m: np32(wl.g[m]) for m in wl.ms}
    return oracle.verify_round(
        oracle_cfg(wl), wl.parents, wl.L, _LazyNp(wl.Q), comp, wl.sel, _LazyNp(wl.rawK),
        _LazyNp(wl.rawV), _LazyNp(wl.treeK), _LazyNp(wl.treeV), g, wl.draft, wl.target,
        requests=requests, with_refresh=with_refresh)


class _LazyNp:
    """Index a stored torch tensor request by request as float32 numpy (bounded memory)."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, b):
        return np32(self.t[b])


def close(got, want, tol, what):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    err = np.abs(got - want)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    mx = float(err.max()) if err.size else 0.0
    mean = float(err.mean()) if err.size else 0.0
    assert mx <= tol["max_abs"], f"{what}: max-abs error {mx:.3g} > {tol['max_abs']}"
    assert mean <= tol["mean_abs"], f"{what}: mean-abs error {mean:.3g} > {tol['mean_abs']}"
    return mx, mean


def to_u64(t):
    return t.detach().cpu().numpy().astype(np.int64).view(np.uint64)


def gpu_round(wl, attn_kernel=_lib.TV_ATTN_AUTO, comp=None, commit=True, stage_chain=0):
    """Upload the workload, seed the compressed prefix (oracle-made unless given), run one round."""
    shape = engine.shape_for(wl, attn_kernel, stage_chain=stage_chain)
    st = engine.alloc_state(wl)
    rb = engine.alloc_round(wl, shape)
    if comp is not None:
        upload_prefix(wl, st, comp)
    st0 = st.clone()
    engine.verify_round(shape, st, rb, commit=commit)
    torch.cuda.synchronize()
    return shape, st0, st, rb


def check_round(wl, res, st0, st, rb, requests, staged=False):
    """Compare one GPU round against the oracle results ``res`` for the listed requests.

    ``staged``: the round ran with tv_shape.stage_chain = 1, so raw rows at and past the new
    length and C4 entries at and past L_new // 4 may hold staged rows of the cached chain; only
    the state a later call can see (rows before L_new, entries before L_new // m) is compared."""
    tol = TOL[wl.dtype]
    status = int(rb.status.item())
    assert status == 0, f"device status {status}"
    anc = to_u64(rb.anc)
    vis = {4: to_u64(rb.vis4), 128: to_u64(rb.vis128)}
    depth = rb.depth.cpu().numpy()
    raw_lo = rb.raw_lo.cpu().numpy()
    O = np32(rb.O)
    lse = rb.lse.cpu().numpy()
    acc = rb.accept_len.cpu().numpy()
    path = rb.path.cpu().numpy()
    bonus = rb.bonus.cpu().numpy()
    committed = rb.committed.cpu().numpy()
    L_new = st.L.cpu().numpy()
    scr = {4: (np32(rb.scrK4), np32(rb.scrV4)), 128: (np32(rb.scrK128), np32(rb.scrV128))}
    errs = []
    for b in requests:
        r = res[b]
        plan = r["plan"]
        # integers: bit-exact
        assert [int(x) for x in anc[b]] == plan.anc, f"anc mismatch, request {b}"
        assert depth[b].tolist() == plan.depth
        assert raw_lo[b].tolist() == plan.raw_lo
        for m in wl.ms:
            assert [int(x) for x in vis[m][b]] == plan.scr_vis[m], f"scr_vis{m}, request {b}"
        assert int(acc[b]) == r["accept_len"]
        n = r["accept_len"]
        assert path[b][:n].tolist() == r["path"] and np.all(path[b][n:] == -1)
        assert int(bonus[b]) == r["bonus"]
        # scratch pad: the oracle's entries where a node closes a block, zeros elsewhere
        for m in wl.ms:
            want_k = np.zeros((wl.D, wl.d))
            want_v = np.zeros((wl.D, wl.d))
            for (mm, u), (ck, cv) in r["scratch"].items():
                if mm == m:
                    want_k[u], want_v[u] = ck, cv
            close(scr[m][0][b], want_k, tol, f"scratch K{m} request {b}")
            close(scr[m][1][b], want_v, tol, f"scratch V{m} request {b}")
        # attention
        errs.append(close(O[b], r["O"], tol, f"O request {b}"))
        lerr = float(np.abs(lse[b] - r["LSE"]).max())
        assert lerr <= tol["lse"], f"LSE request {b}: {lerr:.3g}"
        if "L_new" in r:
            assert int(L_new[b]) == r["L_new"]
            assert committed[b].tolist() == r["committed"].tolist()
            L0 = int(wl.L[b])
            rows_k = np32(st.rawK[b, L0:r["L_new"]])
            rows_v = np32(st.rawV[b, L0:r["L_new"]])
            assert np.array_equal(rows_k, r["raw_rows"][0]), f"raw K rows request {b}"
            assert np.array_equal(rows_v, r["raw_rows"][1]), f"raw V rows request {b}"
            # untouched raw rows before L and after L_new
            assert torch.equal(st.rawK[b, :L0], st0.rawK[b, :L0])
            if not staged:
                assert torch.equal(st.rawK[b, r["L_new"]:], st0.rawK[b, r["L_new"]:])
            for (m, j), (ck, cv) in r["entries"].items():
                dk = st.c4K if m == 4 else st.c128K
                dv = st.c4V if m == 4 else st.c128V
                close(np32(dk[b, j]), ck, tol, f"committed C{m}[{j}] K request {b}")
                close(np32(dv[b, j]), cv, tol, f"committed C{m}[{j}] V request {b}")
            for m in wl.ms:
                ck_new = st.c4K if m == 4 else st.c128K
                ck_old = st0.c4K if m == 4 else st0.c128K
                written = {j for (mm, j) in r["entries"] if mm == m}
                end = r["L_new"] // m if (staged and m == 4) else ck_new.shape[1]
                keep = [j for j in range(end) if j not in written]
                assert torch.equal(ck_new[b, keep], ck_old[b, keep]), f"C{m} rows changed, request {b}"
    return errs

"""ctypes binding of libtreeverify.so (argument marshalling only).

Every function here forwards torch tensors' device pointers and the current CUDA stream to the
C entry point of the same name declared in ``include/treeverify.h``; all arithmetic runs in the
library's CUDA kernels.  A missing or unloadable library raises ``RuntimeError``: there is no
fallback implementation.
"""

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# TV_LIB_CHECKED=1 loads the bounds-checked debug build of the same library instead
LIB_PATH = os.path.join(_PKG, "libtreeverify_checked.so" if os.environ.get("TV_LIB_CHECKED") == "1"
                        else "libtreeverify.so")

TV_OK = 0
TV_ERR = {
    -1: "TV_ERR_ARG", -2: "TV_ERR_SHAPE", -3: "TV_ERR_BAD_TREE", -4: "TV_ERR_CAPACITY",
    -5: "TV_ERR_DTYPE", -6: "TV_ERR_CUDA", -7: "TV_ERR_WORKSPACE", -8: "TV_ERR_TIMEOUT",
    -9: "TV_ERR_SELECTION", -10: "TV_ERR_BOUNDS",
}
TV_TAIL_WINDOW, TV_TAIL_REMAINDER = 0, 1
TV_COMP_C4, TV_COMP_C128 = 1, 2
TV_F32, TV_BF16 = 0, 1
TV_ATTN_AUTO, TV_ATTN_SIMT, TV_ATTN_TCGEN05 = 0, 1, 2

EXPORTS = (
    "tv_version", "tv_status_string", "tv_last_error_string", "tv_workspace_size",
    "tv_attn_kernel_for",
    "tv_build_ancestor_mask", "tv_prefill_compress", "tv_branch_compress",
    "tv_tree_verify_attn", "tv_accept_walk", "tv_refresh_commit", "tv_tree_verify_attn_noalloc",
    "tv_indexer_workspace_size", "tv_indexer_topk", "tv_debug_attn_timeout", "tv_noalloc_prepare",
)


class tv_shape(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("D", ctypes.c_int32), ("H", ctypes.c_int32),
        ("d", ctypes.c_int32), ("W", ctypes.c_int32), ("tail_mode", ctypes.c_int32),
        ("comp_mask", ctypes.c_int32), ("dtype", ctypes.c_int32), ("n_sel", ctypes.c_int32),
        ("attn_kernel", ctypes.c_int32), ("raw_cap", ctypes.c_int64), ("c4_cap", ctypes.c_int64),
        ("c128_cap", ctypes.c_int64), ("page_tokens", ctypes.c_int32),
        ("max_pages", ctypes.c_int32), ("n_pool_pages", ctypes.c_int32),
        ("stage_chain", ctypes.c_int32), ("page_table", ctypes.c_void_p),
    ]


class TreeVerifyError(RuntimeError):
    def __init__(self, fn, code, message):
        super().__init__(f"{fn}: {TV_ERR.get(code, code)}: {message}")
        self.code = code


_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_SHAPE = ctypes.POINTER(tv_shape)
_SIGS = {
    "tv_version": ([], ctypes.c_char_p),
    "tv_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "tv_last_error_string": ([], ctypes.c_char_p),
    "tv_workspace_size": ([_SHAPE], ctypes.c_size_t),
    "tv_attn_kernel_for": ([_SHAPE], ctypes.c_int),
    "tv_build_ancestor_mask": ([_SHAPE] + [_P] * 8 + [_P], ctypes.c_int),
    "tv_prefill_compress": ([_SHAPE] + [_P] * 10 + [_P], ctypes.c_int),
    "tv_branch_compress": ([_SHAPE] + [_P] * 15 + [_P], ctypes.c_int),
    "tv_tree_verify_attn": ([_SHAPE] + [_P] * 19 + [ctypes.c_float, _P, _P, _P, ctypes.c_size_t,
                                                    _P, _P], ctypes.c_int),
    "tv_tree_verify_attn_noalloc": ([_SHAPE] + [_P] * 19 + [ctypes.c_float, _P, _P, _P, _P],
                                    ctypes.c_int),
    "tv_accept_walk": ([_SHAPE] + [_P] * 7 + [_P], ctypes.c_int),
    "tv_refresh_commit": ([_SHAPE] + [_P] * 18 + [_P], ctypes.c_int),
    "tv_indexer_workspace_size": ([_SHAPE], ctypes.c_size_t),
    "tv_indexer_topk": ([_SHAPE, ctypes.c_int] + [_P] * 5 + [ctypes.c_size_t, _P, _P],
                        ctypes.c_int),
    "tv_noalloc_prepare": ([], ctypes.c_int),
    "tv_debug_attn_timeout": ([ctypes.c_int64, ctypes.c_int32], ctypes.c_int),
}


def load():
    """Load (once) and return the library; raise if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libtreeverify.so not found at {LIB_PATH}: build it first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in _SIGS.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
        return _lib


def version():
    return load().tv_version().decode()


def make_shape(*, B, D, H, d, W=0, tail_mode=TV_TAIL_WINDOW, comp_mask=TV_COMP_C4 | TV_COMP_C128,
               dtype=TV_BF16, n_sel=0, attn_kernel=TV_ATTN_AUTO, raw_cap=0, c4_cap=0, c128_cap=0,
               page_tokens=0, max_pages=0, n_pool_pages=0, page_table=None, stage_chain=0):
    """``page_table``: a CUDA int32 tensor [B][max_pages] (paged pools only); the shape keeps its
    device address, so the tensor must outlive the shape's use.  ``stage_chain``: 1 stages the
    cached chain's raw rows and C4 entries in tv_branch_compress and skips them in
    tv_refresh_commit."""
    pt = None if page_table is None else _p(page_table).value
    return tv_shape(B, D, H, d, W, tail_mode, comp_mask, dtype, n_sel, attn_kernel, raw_cap,
                    c4_cap, c128_cap, page_tokens, max_pages, n_pool_pages, stage_chain, pt)


def _p(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor or None")
    if not t.is_cuda:
        raise ValueError("tensor arguments must live on the CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn, rc):
    if rc != TV_OK:
        msg = load().tv_last_error_string().decode()
        raise TreeVerifyError(fn, rc, msg)


def tv_workspace_size(shape):
    return int(load().tv_workspace_size(ctypes.byref(shape)))


def tv_attn_kernel_for(shape):
    rc = int(load().tv_attn_kernel_for(ctypes.byref(shape)))
    if rc < 0:
        _check("tv_attn_kernel_for", rc)
    return rc


def tv_build_ancestor_mask(shape, parents, L, anc, depth, raw_lo, scr_vis4, scr_vis128, status,
                           stream=None):
    rc = load().tv_build_ancestor_mask(ctypes.byref(shape), _p(parents), _p(L), _p(anc), _p(depth),
                                       _p(raw_lo), _p(scr_vis4), _p(scr_vis128), _p(status),
                                       _stream(stream))
    _check("tv_build_ancestor_mask", rc)


def tv_prefill_compress(shape, rawK, rawV, L, g4, g128, c4K, c4V, c128K, c128V, status,
                        stream=None):
    rc = load().tv_prefill_compress(ctypes.byref(shape), _p(rawK), _p(rawV), _p(L), _p(g4),
                                    _p(g128), _p(c4K), _p(c4V), _p(c128K), _p(c128V), _p(status),
                                    _stream(stream))
    _check("tv_prefill_compress", rc)


def tv_branch_compress(shape, rawK, rawV, c4K, c4V, L, treeK, treeV, parents, g4, g128, scrK4,
                       scrV4, scrK128, scrV128, status, stream=None):
    rc = load().tv_branch_compress(ctypes.byref(shape), _p(rawK), _p(rawV), _p(c4K), _p(c4V),
                                   _p(L), _p(treeK), _p(treeV), _p(parents), _p(g4), _p(g128),
                                   _p(scrK4), _p(scrV4), _p(scrK128), _p(scrV128), _p(status),
                                   _stream(stream))
    _check("tv_branch_compress", rc)


def tv_tree_verify_attn(shape, Q, c4K, c4V, sel, c128K, c128V, rawK, rawV, L, treeK, treeV, anc,
                        raw_lo, scr_vis4, scr_vis128, scrK4, scrV4, scrK128, scrV128, scale, O,
                        lse, workspace, status, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().tv_tree_verify_attn(ctypes.byref(shape), _p(Q), _p(c4K), _p(c4V), _p(sel),
                                    _p(c128K), _p(c128V), _p(rawK), _p(rawV), _p(L), _p(treeK),
                                    _p(treeV), _p(anc), _p(raw_lo), _p(scr_vis4), _p(scr_vis128),
                                    _p(scrK4), _p(scrV4), _p(scrK128), _p(scrV128),
                                    ctypes.c_float(scale), _p(O), _p(lse), _p(workspace),
                                    ctypes.c_size_t(ws_bytes), _p(status), _stream(stream))
    _check("tv_tree_verify_attn", rc)


def tv_tree_verify_attn_noalloc(shape, Q, c4K, c4V, sel, c128K, c128V, rawK, rawV, L, treeK,
                                treeV, anc, raw_lo, scr_vis4, scr_vis128, scrK4, scrV4, scrK128,
                                scrV128, scale, O, lse, status, stream=None):
    """tv_tree_verify_attn for callers that cannot allocate: no workspace argument; the library's
    built-in scratch holds the split-KV partials (see include/treeverify.h)."""
    rc = load().tv_tree_verify_attn_noalloc(
        ctypes.byref(shape), _p(Q), _p(c4K), _p(c4V), _p(sel), _p(c128K), _p(c128V), _p(rawK),
        _p(rawV), _p(L), _p(treeK), _p(treeV), _p(anc), _p(raw_lo), _p(scr_vis4), _p(scr_vis128),
        _p(scrK4), _p(scrV4), _p(scrK128), _p(scrV128), ctypes.c_float(scale), _p(O), _p(lse),
        _p(status), _stream(stream))
    _check("tv_tree_verify_attn_noalloc", rc)


def tv_accept_walk(shape, parents, draft, target, accept_len, path, bonus, status, stream=None):
    rc = load().tv_accept_walk(ctypes.byref(shape), _p(parents), _p(draft), _p(target),
                               _p(accept_len), _p(path), _p(bonus), _p(status), _stream(stream))
    _check("tv_accept_walk", rc)


def tv_refresh_commit(shape, parents, accept_len, path, treeK, treeV, scrK4, scrV4, scrK128,
                      scrV128, rawK, rawV, c4K, c4V, c128K, c128V, L, committed_pos, status,
                      stream=None):
    rc = load().tv_refresh_commit(ctypes.byref(shape), _p(parents), _p(accept_len), _p(path),
                                  _p(treeK), _p(treeV), _p(scrK4), _p(scrV4), _p(scrK128),
                                  _p(scrV128), _p(rawK), _p(rawV), _p(c4K), _p(c4V), _p(c128K),
                                  _p(c128V), _p(L), _p(committed_pos), _p(status), _stream(stream))
    _check("tv_refresh_commit", rc)


def tv_noalloc_prepare():
    """Load the library's device code (with the 32 MiB built-in scratch) on the current device."""
    _check("tv_noalloc_prepare", load().tv_noalloc_prepare())


def tv_indexer_workspace_size(shape):
    return int(load().tv_indexer_workspace_size(ctypes.byref(shape)))


def tv_indexer_topk(shape, d_idx, q_idx, k_idx, L, sel, workspace, status, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().tv_indexer_topk(ctypes.byref(shape), ctypes.c_int(d_idx), _p(q_idx), _p(k_idx),
                                _p(L), _p(sel), _p(workspace), ctypes.c_size_t(ws_bytes),
                                _p(status), _stream(stream))
    _check("tv_indexer_topk", rc)


def tv_debug_attn_timeout(timeout_ns, withhold_tile):
    """Testing aid: the wait bound and a withheld KV tile of later tensor-core attention calls."""
    _check("tv_debug_attn_timeout", load().tv_debug_attn_timeout(int(timeout_ns), int(withhold_tile)))

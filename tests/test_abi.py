"""The C-ABI library loads, exports every symbol include/treeverify.h declares, and its host-side
validation rejects bad arguments -- all without touching a GPU."""

import ctypes
import os
import re

import pytest

from tree_speculative_verify_gb300 import _lib, build as tvbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "treeverify.h")


@pytest.fixture(scope="module")
def lib():
    tvbuild.build()
    return _lib.load()


def _declarations():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    decls = {}
    for m in re.finditer(r"^\s*[\w\s\*]+?\b(tv_\w+)\s*\(([^;]*?)\)\s*;", text, flags=re.M | re.S):
        args = m.group(2).strip()
        n = 0 if args in ("", "void") else args.count(",") + 1
        decls[m.group(1)] = n
    return decls


def test_header_declares_the_entry_points():
    decls = _declarations()
    for name in _lib.EXPORTS:
        assert name in decls, name
    assert set(decls) == set(_lib.EXPORTS)


def test_header_compiles_as_c_and_cxx(tmp_path):
    # the boundary is plain C: the header alone compiles as C11 and as C++17, warnings as errors
    import shutil
    import subprocess
    src = tmp_path / "use.c"
    src.write_text('#include "treeverify.h"\n'
                   'int probe(tv_shape* s) { return (int)tv_workspace_size(s) + s->B; }\n')
    for cc, std in (("gcc", "-std=c11"), ("g++", "-std=c++17")):
        if shutil.which(cc) is None:
            pytest.skip(f"{cc} not installed")
        args = [cc, std, "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
                "-I", os.path.dirname(HEADER)]
        if cc == "g++":
            args += ["-x", "c++"]
        r = subprocess.run(args + [str(src)], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_every_declared_symbol_is_exported(lib):
    for name in _declarations():
        assert hasattr(lib, name), name


def test_binding_signatures_match_header(lib):
    decls = _declarations()
    for name, n in decls.items():
        assert len(_lib._SIGS[name][0]) == n, (name, len(_lib._SIGS[name][0]), n)


def test_version_and_status_strings(lib):
    assert "treeverify" in _lib.version()
    assert lib.tv_status_string(-3) == b"TV_ERR_BAD_TREE"
    assert lib.tv_status_string(0) == b"TV_OK"


def test_struct_layout_matches_c():
    assert ctypes.sizeof(_lib.tv_shape) == 10 * 4 + 3 * 8 + 4 * 4 + 8


def _shape(**kw):
    base = dict(B=2, D=8, H=64, d=512, W=128, raw_cap=1000, c4_cap=260, c128_cap=9)
    base.update(kw)
    return _lib.make_shape(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(D=0), -2), (dict(D=65), -2), (dict(d=12), -2), (dict(d=1024), -2), (dict(H=0), -2),
    (dict(tail_mode=7), -1), (dict(comp_mask=0), -1), (dict(dtype=3), -1), (dict(B=-1), -2),
    (dict(n_sel=5, comp_mask=2), -1), (dict(attn_kernel=9), -1), (dict(raw_cap=-1), -2),
])
def test_host_validation_rejects_bad_shapes(lib, kw, code):
    s = _shape(**kw)
    rc = lib.tv_accept_walk(ctypes.byref(s), None, None, None, None, None, None, None, None)
    assert rc == code
    assert lib.tv_last_error_string() != b""
    assert lib.tv_workspace_size(ctypes.byref(s)) == 0


def test_null_pointers_rejected_before_any_launch(lib):
    s = _shape()
    rc = lib.tv_build_ancestor_mask(ctypes.byref(s), None, None, None, None, None, None, None,
                                    None, None)
    assert rc == -1 and b"null" in lib.tv_last_error_string()
    rc = lib.tv_refresh_commit(ctypes.byref(s), *([None] * 19))
    assert rc == -1


def test_misaligned_q_or_o_rejected_before_any_launch(lib):
    # stand-in device addresses: validation returns before anything touches them
    s = _shape()
    ok = ctypes.c_void_p(1 << 20)
    ws_bytes = lib.tv_workspace_size(ctypes.byref(s))

    def call(Q, O):
        return lib.tv_tree_verify_attn(ctypes.byref(s), Q, *([ok] * 18), ctypes.c_float(0.05), O,
                                       ok, ok, ws_bytes, ok, None)

    rc = call(ok, ctypes.c_void_p((1 << 20) + 8))
    assert rc == -1 and b"16-byte aligned" in lib.tv_last_error_string()
    rc = call(ctypes.c_void_p((1 << 20) + 2), ok)
    assert rc == -1 and b"16-byte aligned" in lib.tv_last_error_string()


def test_empty_batch_is_a_no_op(lib):
    s = _shape(B=0)
    assert lib.tv_accept_walk(ctypes.byref(s), None, None, None, None, None, None, None, None) == 0
    assert lib.tv_workspace_size(ctypes.byref(s)) == 0


def test_workspace_size_grows_with_batch(lib):
    a = lib.tv_workspace_size(ctypes.byref(_shape(B=2)))
    b = lib.tv_workspace_size(ctypes.byref(_shape(B=4)))
    assert 0 < a < b and a % 256 == 0


def test_indexer_validation(lib):
    s = _shape(n_sel=64)
    rc = lib.tv_indexer_topk(ctypes.byref(s), 12, None, None, None, None, None, 0, None, None)
    assert rc == -2                                           # d_idx not a multiple of 8
    s0 = _shape(n_sel=0)
    rc = lib.tv_indexer_topk(ctypes.byref(s0), 64, None, None, None, None, None, 0, None, None)
    assert rc == -1                                           # no selection size
    rc = lib.tv_indexer_topk(ctypes.byref(s), 64, None, None, None, None, None, 0, None, None)
    assert rc == -1                                           # null inputs
    assert lib.tv_indexer_workspace_size(ctypes.byref(s)) == 2304         # 2 x 260 x 4, to 256


def test_paging_validation(lib):
    # page size not a multiple of 512; capacities inconsistent with the pages; no page table
    s = _shape(page_tokens=300, max_pages=4, n_pool_pages=8)
    assert lib.tv_accept_walk(ctypes.byref(s), *([None] * 8)) == -2
    s = _shape(page_tokens=512, max_pages=2, n_pool_pages=8, raw_cap=1024, c4_cap=256, c128_cap=9)
    assert lib.tv_accept_walk(ctypes.byref(s), *([None] * 8)) == -2
    s = _shape(page_tokens=512, max_pages=2, n_pool_pages=8, raw_cap=1024, c4_cap=256, c128_cap=8)
    assert lib.tv_accept_walk(ctypes.byref(s), *([None] * 8)) == -1      # page_table is null
    s.stage_chain = 2
    assert lib.tv_workspace_size(ctypes.byref(s)) == 0

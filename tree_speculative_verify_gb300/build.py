"""Build libtreeverify.so in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` file is compiled to an object file in parallel, then the objects are linked
into ``tree_speculative_verify_gb300/libtreeverify.so``.  The CUDA runtime is linked statically,
so the library only needs the NVIDIA driver at run time.  A rebuild is skipped when the library
is newer than every source and header.
"""

import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libtreeverify.so")
# the bounds-checked debug build (-DTV_CHECK_BOUNDS): every checked global index that fails its
# range check records TV_ERR_BOUNDS and skips the access (see tv_common.cuh)
LIB_CHECKED = os.path.join(PKG, "libtreeverify_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I" + INCLUDE, "-I" + CSRC]


def nvcc_path():
    cand = shutil.which("nvcc")
    if cand:
        return cand
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libtreeverify")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date(lib=LIB):
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force=False, verbose=False, extra_flags=(), checked=False):
    """Compile and link the library (checked: the bounds-checked debug build, a separate file);
    returns its path."""
    lib = LIB_CHECKED if checked else LIB
    if not force and up_to_date(lib):
        return lib
    nvcc = nvcc_path()
    objdir = os.path.join(BUILD, "checked") if checked else BUILD
    os.makedirs(objdir, exist_ok=True)
    srcs = _sources()
    flags = list(extra_flags) + (["-DTV_CHECK_BOUNDS"] if checked else [])

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src).replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    workers = min(len(srcs), os.cpu_count() or 4)
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    force = "--force" in sys.argv
    verbose = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []
    print(build(force=force or bool(extra), verbose=verbose or bool(extra), extra_flags=extra,
                checked="--checked" in sys.argv))

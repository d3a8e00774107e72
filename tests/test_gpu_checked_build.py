"""The bounds-checked debug build (-DTV_CHECK_BOUNDS): every checked global index of the
tensor-core attention's producer and epilogue and of the persistent-row addressing is range-checked
on the device (a violation records TV_ERR_BOUNDS and skips the access).  Representative parity
cases -- contiguous and paged pools, split KV, the sparse selection path, staging and several
rounds -- run against that build in a child process and must pass with a clean status word."""

import os
import subprocess
import sys

import pytest

from tree_speculative_verify_gb300 import build as tvbuild

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

CASES = [
    "test_gpu_parity.py::test_small_bf16_full_size",
    "test_gpu_parity.py::test_serving_reduced_batch",
    "test_gpu_parity.py::test_long_context_reduced",
    "test_gpu_parity.py::test_split_kv_with_empty_chunks",
    "test_gpu_parity.py::test_short_prefixes",
    "test_gpu_parity.py::test_two_rounds_in_a_row",
    "test_gpu_paged.py",
    "test_gpu_stage_chain.py::test_staged_rounds_equal_unstaged_bit_for_bit",
    "test_gpu_compress.py",
]


def test_parity_cases_pass_under_the_bounds_checked_build():
    tvbuild.build(checked=True)
    env = dict(os.environ, TV_LIB_CHECKED="1")
    probe = subprocess.run([sys.executable, "-c", "from tree_speculative_verify_gb300 import _lib; "
                            "print(_lib.LIB_PATH)"], cwd=ROOT, env=env, capture_output=True,
                           text=True, timeout=300)
    assert probe.stdout.strip().endswith("libtreeverify_checked.so"), probe.stdout + probe.stderr
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider"]
    cmd += [os.path.join(HERE, c) for c in CASES]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert "treeverify bounds check" not in r.stdout + r.stderr, tail

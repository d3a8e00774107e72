"""GB300-native target-verify path of tree-structured speculative decoding over
online-compressed (C4 / C128) attention.

The compute lives in ``libtreeverify.so`` (C ABI, ``include/treeverify.h``, CUDA kernels for
sm_103a).  This package is its thin Python binding: functions with the C entry points' names
(``tv_build_ancestor_mask``, ``tv_prefill_compress``, ``tv_branch_compress``,
``tv_tree_verify_attn``, ``tv_accept_walk``, ``tv_refresh_commit``, ``tv_workspace_size``) that
marshal torch tensors' device pointers, plus ``engine`` (device buffers, the five-call round)
and ``workloads`` (seeded synthetic inputs).  The library is loaded on first use; a missing
library raises ``RuntimeError``.
"""

from ._lib import (  # noqa: F401
    TV_ATTN_AUTO, TV_ATTN_SIMT, TV_ATTN_TCGEN05, TV_BF16, TV_COMP_C128, TV_COMP_C4, TV_F32,
    TV_TAIL_REMAINDER, TV_TAIL_WINDOW, TreeVerifyError, load, make_shape, tv_accept_walk, tv_attn_kernel_for,
    tv_branch_compress, tv_build_ancestor_mask, tv_prefill_compress, tv_refresh_commit, tv_shape,
    tv_tree_verify_attn, tv_workspace_size, version,
)

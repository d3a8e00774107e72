"""CPU oracle for tree-structured speculative verification over online-compressed attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package: only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may use it.

The oracle is a plain, slow, fp64 numpy restatement of what the target-verify path computes,
written from the report "Adapting Tree-Structured Speculative Decoding to DeepSeek-V4 for
Efficient Inference" (arXiv 2609.24698), cited below as [TSD-V4].  The report lost its section
headings when it was scraped; the section numbers used here are inferred from its in-text
cross-references (§2.2 CSA/HCA compression, §3.1-3.2 branch-aware causality and isolation,
§4.1 the three-stage speculative forward and the verification plan, §4.2 scratch pad and
state refresh, §4.3 optimisations, §5.1 the ``sN_kK_dD`` naming).

Every stored floating-point value (compressed entries, persistent or in the scratch pad) is
rounded to the cache's storage dtype with round-to-nearest-even, exactly as the GPU path
stores it; everything else is computed in fp64.

Modules
-------
storage   fp64 -> bf16 / fp32 rounding of stored values
compress  the per-block gated-sum compressor (C4 and C128)
plan      parent array -> ancestor masks, depths, positions, window bounds, scratch visibility
verify    branch-aware causal attention of every tree node over its visible set
accept    the greedy acceptance walk
refresh   accepted-path commit of raw K/V and completed compressed blocks
round     one full verify round: the five steps above in order
indexer   top-k selection of persistent C4 entries by an fp32 indexer score (sparse C4 path)

Parity status: every function here is pinned by the ``-m "not gpu"`` tests
(``tests/test_oracle_*.py``) against brute force, closed forms, special cases or library
routines; nothing is "parity unpinned".
"""

from .storage import round_to_storage, to_f64
from .compress import gated_block_sum, compress_blocks, compress_prefix
from .plan import build_plan, Plan
from .verify import (
    VerifyConfig,
    path_to_root,
    sequence_row,
    scratch_entries,
    visible_set,
    tree_verify_attn_request,
)
from .accept import accept_walk
from .refresh import refresh_commit_request
from .round import verify_round
from .indexer import index_scores, topk_ascending, indexer_select

__all__ = [
    "round_to_storage",
    "to_f64",
    "gated_block_sum",
    "compress_blocks",
    "compress_prefix",
    "build_plan",
    "Plan",
    "VerifyConfig",
    "path_to_root",
    "sequence_row",
    "scratch_entries",
    "visible_set",
    "tree_verify_attn_request",
    "accept_walk",
    "refresh_commit_request",
    "verify_round",
    "index_scores",
    "topk_ascending",
    "indexer_select",
]

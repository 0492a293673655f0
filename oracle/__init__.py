"""fp64 CPU oracle for block-hybrid attention (test infrastructure only).

This package is the checker, not the product. Only the tests, the smoke check
of ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it.
It shares no code with the CUDA library: no kernels, headers, helpers,
constants or pre/post-processing. Inputs reach it as plain numpy arrays.
"""

from .block_hybrid import (  # noqa: F401
    MERGE_CONVEX,
    MERGE_SHARED_NORM,
    attend,
    attend_gqa,
    attend_bruteforce,
    commit,
    feature_map,
    gather_pages,
    kv_head,
    prefill,
    prefill_attend,
    sigmoid,
    softmax_kv_attend,
    softmax_kv_attend_paged,
)

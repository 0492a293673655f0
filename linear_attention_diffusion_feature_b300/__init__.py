"""Block-hybrid attention for blockwise diffusion language models on B300.

Exact bidirectional softmax within the active block, a Hedgehog linear read
of a fixed-size per-head state for all committed blocks, and a gated merge,
as hand-written sm_103a CUDA kernels behind the C ABI of ``libhb.so``
(``include/hb.h``). This package is the Python binding of that library.
"""

from .hb import (  # noqa: F401
    DTYPE_BF16,
    DTYPE_FP32,
    MERGE_CONVEX,
    MERGE_SHARED_NORM,
    Config,
    HBError,
    hb_block_attend,
    hb_block_attend_commit,
    hb_block_attend_commit_layers,
    hb_block_attend_commit_s16,
    hb_block_attend_ex,
    hb_commit_block,
    hb_feature_map,
    hb_get_device_status,
    hb_set_wait_limit,
    hb_prefill_attend,
    hb_prefill_attend_ex,
    hb_prefill_state,
    hb_prefill_state_noalloc,
    hb_prefill_workspace_size,
    hb_softmax_kv_attend,
    hb_softmax_kv_attend_paged,
    hb_softmax_kv_workspace_size,
    hb_block_attend_s16,
    hb_block_attend_s8,
    hb_state_copy,
    hb_state_to_bf16,
    hb_state_to_fp8,
    hb_state_zero,
    hb_status_string,
)

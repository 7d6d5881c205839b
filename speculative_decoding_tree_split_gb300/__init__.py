"""Split tree attention for speculative-decoding verification on GB300 (sm_103a).

The work runs in ``libtreeattn.so`` (hand-written CUDA for sm_103a behind the
C ABI in ``include/tree_attn.h``); this package is its thin Python binding.

    mask = mask_build(parents)                     # uint64 ancestor bits [T]
    out, lse = verify(q, k_pages, v_pages, block_table, seq_lens,
                      tree_k, tree_v, mask, workspace=ws)

``build()`` compiles the library in place with nvcc.
"""
from ._build import build, LIB as LIB_PATH  # noqa: F401
from ._lib import (  # noqa: F401
    ERRORS,
    EXPORTED,
    MAX_T,
    STATUS_BAD_PAGE,
    STATUS_BAD_PARENT,
    STATUS_BAD_SEQ_LEN,
    STATUS_TIMEOUT,
    STATUS_BAD_PATH,
    TreeAttnError,
    load,
    mask_build,
    mask_build_batched,
    plan,
    prefix_pass,
    suffix_merge,
    verify,
    verify_batched,
    verify_paged_tree,
    verify_tree,
    greedy_accept,
    dense_cols_for,
    dense_mask_build,
    verify_dense,
    kv_commit,
    accept_commit,
    version,
    workspace_size,
    set_wait_limit_ns,
    set_early_prefix_loads,
    DEFAULT_WAIT_NS,
)

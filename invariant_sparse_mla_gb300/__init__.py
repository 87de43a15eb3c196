"""GB300-native deterministic sparse top-k and sparse MLA attention.

The compute lives in hand-written sm_103a CUDA kernels behind the C ABI of
``include/ds_sparse_mla.h`` (``libds_sparse_mla.so``, built in-tree by
``invariant_sparse_mla_gb300.build``). This package only marshals torch
tensors and the current stream into those calls.
"""

from ._native import (  # noqa: F401
    DSError,
    DEVERR_IDX,
    DEVERR_PAGE,
    DEVERR_ROWREQ,
    DEVERR_TIMEOUT,
    EXPORTED,
    attention_workspace_size,
    indexer_logits,
    kv_cache_write,
    last_error,
    lib,
    sparse_mla_decode,
    sparse_mla_decode_swa,
    sparse_mla_prefill,
    supported_config,
    swa_workspace_size,
    topk_per_row,
    topk_workspace_size,
)

"""GB300 (sm_103a) batched, ragged, exact per-row top-k over FP32 indexer scores.

Every call is enqueued on a CUDA stream and computed entirely by the library's
CUDA kernels (``_build/libtopk_indexer.so``):

* :func:`topk_ragged` - indices of each row's k largest scores, ``-1`` past
  the row's length;
* :func:`topk_paged` - the same indices mapped through a page table;
* :func:`topk_select_bf16` - the same selection over bfloat16 scores (rows of
  at most 16384);
* :func:`amax8_varlen`, :func:`sort_candidate_blocks` - the two-level
  indexer's block-max keys and sorted candidate block table;
* :func:`topk_select_ex` - diagnostics: a forced internal path, path counters;
  :func:`max_active_clusters` - the CUDA driver's cluster residency per size.

PyTorch only provides device memory and streams.
"""

from ._binding import (  # noqa: F401
    DEVICE_ERROR_INDEX,
    LIB_PATH,
    NUM_COUNTERS,
    TOPK_MAX_K,
    Counter,
    Status,
    TopkError,
    amax8_varlen,
    load_library,
    max_active_clusters,
    raw_library,
    sort_candidate_blocks,
    topk_paged,
    topk_ragged,
    topk_select_bf16,
    topk_select_ex,
    workspace_bytes,
)

__all__ = ["topk_ragged", "topk_paged", "topk_select_ex", "topk_select_bf16", "workspace_bytes",
           "amax8_varlen", "sort_candidate_blocks", "max_active_clusters", "TopkError",
           "Status", "Counter",
           "load_library", "raw_library", "LIB_PATH", "TOPK_MAX_K", "NUM_COUNTERS",
           "DEVICE_ERROR_INDEX"]

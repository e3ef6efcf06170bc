"""Quest decode-time hot path for GB300 (sm_103a): paged fp16 KV cache with per-page key
min/max boxes, query-aware page scoring, per-head top-K page selection and split-K
sparse flash-decode, as a C-ABI library (``libquest.so``) with a thin ctypes binding.

The names below mirror the C entry points of ``include/quest.h``.
"""
from ._lib import (  # noqa: F401
    EXPORTS, HEAD_DIM, QUEST_DEBUG_WITHHOLD_SELECTION, QUEST_ERR_BAD_LENGTH,
    QUEST_ERR_BAD_PAGE, QUEST_ERR_BAD_SELECTION, QUEST_ERR_CUDA, QUEST_ERR_INVALID_ARG,
    QUEST_ERR_TIMEOUT, QUEST_ERR_UNSUPPORTED, QUEST_ERR_WORKSPACE, QUEST_MAX_PAGES, QUEST_OK,
    QUEST_PATH_AUTO, QUEST_PATH_CHAIN, QUEST_PATH_FUSED, QUEST_PATH_STREAM,
    DecodePlan, PagedCache, QuestCacheDesc, QuestError, QuestLayer, QuestOpts, append, build_meta, decode,
    decode_launches, decode_layers, decode_path, decode_step,
    dense_decode, estimate, estimate_heads, load, opts, prefill, read_status, sparse_decode, topk, workspace,
    workspace_init, workspace_size,
)

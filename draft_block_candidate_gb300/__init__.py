"""GB300-native (sm_103a) LiLiCorr draft-time rerank.

The CUDA library (liblilicorr.so, built in-tree by build.build()) holds the whole path;
this package marshals arguments to its C ABI.
"""
from .api import (  # noqa: F401
    LilicorrError,
    Weights,
    device_error,
    diag_wait_timeout,
    greedy_walk,
    viterbi,
    launch_count,
    lm_head_topk_lse,
    lm_head_workspace_bytes,
    rerank,
    rerank_host,
    rerank_host_workspace,
    sample_walk,
    stage_timing,
    stage_times,
    topk_lse,
    topk_lse_merge,
    topk_lse_shard,
    topk_lse_workspace,
)
from ._lib import BF16, F32, LIB_PATH  # noqa: F401

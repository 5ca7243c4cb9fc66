"""GB300-native DeepSeek-Sparse-Attention (DSA) layer hot path.

Python face of libdsa (C ABI in include/dsa.h): the causal pooled indexer
with per-query top-k (``dsa_index_topk``) and the sparse attention forward
and backward (``dsa_sparse_attn_fwd`` / ``dsa_sparse_attn_bwd``).  Inputs are
CUDA tensors; every step runs in hand-written sm_103a kernels.
"""
from ._binding import (DSA_ERR_CUDA, DSA_ERR_INTERNAL, DSA_ERR_INVALID_ARG, DSA_ERR_TIMEOUT, DSA_ERR_UNSUPPORTED,
                       DSA_ERR_WORKSPACE, DSA_OK, EXPORTED, LIB_PATH, DsaError, dsa_clear_status, dsa_index_topk,
                       dsa_index_topk_noalloc,
                       dsa_sparse_attn_bwd, dsa_sparse_attn_fwd, dsa_sparse_attn_fwd_tc, dsa_sync_status, index_topk_workspace_size, load,
                       sparse_attn_bwd_workspace_size, version, profile_enable, profile_read, launch_count,
                       launch_count_reset, zigzag_ranges, dsa_index_topk_varlen, dsa_sparse_attn_fwd_varlen,
                       dsa_sparse_attn_bwd_varlen, dsa_sparse_attn_bwd_deterministic,
                       sparse_attn_bwd_deterministic_workspace_size, index_topk_stats, measure_l2, measure_umma, measure_fold, last_kernel_config)

__all__ = ["dsa_index_topk", "dsa_index_topk_noalloc", "dsa_sparse_attn_fwd", "dsa_sparse_attn_fwd_tc", "dsa_sparse_attn_bwd", "dsa_sync_status", "dsa_clear_status",
           "index_topk_workspace_size", "sparse_attn_bwd_workspace_size", "DsaError", "load", "version", "LIB_PATH",
           "EXPORTED", "zigzag_ranges", "dsa_index_topk_varlen", "dsa_sparse_attn_fwd_varlen",
           "dsa_sparse_attn_bwd_varlen", "dsa_sparse_attn_bwd_deterministic",
           "sparse_attn_bwd_deterministic_workspace_size", "profile_enable", "profile_read", "launch_count", "launch_count_reset", "index_topk_stats", "measure_l2", "measure_umma", "measure_fold", "last_kernel_config", "DSA_OK", "DSA_ERR_INVALID_ARG", "DSA_ERR_UNSUPPORTED", "DSA_ERR_WORKSPACE", "DSA_ERR_CUDA",
           "DSA_ERR_TIMEOUT", "DSA_ERR_INTERNAL"]

"""indexer_selected_sparse_block_gb300: indexer-selected block-sparse attention on GB300.

The product is libsfa.so (C ABI in include/sfa.h, CUDA kernels for sm_103a in csrc/); this
package is its Python binding (argument marshalling only), the step runner that chains the
entry points, and the seeded synthetic input generators.
"""
from ._binding import (SFA_BF16, SFA_DEV_BAD_BLOCK, SFA_DEV_BAD_CELL, SFA_DEV_BAD_NSEL,
                       SFA_DEV_BAD_QUERY, SFA_DEV_FP16_RANGE, SFA_DEV_TIMEOUT, SFA_ERR_CUDA,
                       SFA_ERR_INVALID_ARG, SFA_ERR_UNSUPPORTED, SFA_ERR_WORKSPACE, SFA_F32,
                       SFA_OK, SFA_PART_ALL, SFA_PART_SELECTED, SFA_PART_WINDOW, SFA_Q8_0,
                       SFA_REFINE_MAX_BLOCKS, SfaError, kbar_shape, lib,
                       sfa_attend_plan, sfa_attend_workspace_bytes, sfa_combine_attention,
                       sfa_copy_cache_rows, sfa_copy_cache_rows_multi, sfa_dense_attend,
                       sfa_dense_attend_paged,
                       sfa_gather_attend, sfa_gather_attend_noalloc, sfa_gather_attend_paged,
                       sfa_gather_attend_window, sfa_gather_kv_bandwidth, sfa_index_scores,
                       sfa_index_scores_bounded, sfa_index_scores_bounded_i8, k8_shapes,
                       sfa_quantize_pooled_keys_i8, sfa_pool_index_keys, sfa_pool_index_keys_paged,
                       sfa_pool_index_keys_transformed, sfa_q8_0_row_bytes,
                       sfa_quantize_kv_q8_0, sfa_read_device_status, sfa_topk_blocks,
                       sfa_topk_blocks_refine, sfa_topk_refine_workspace_bytes,
                       sfa_topk_workspace_bytes, sfa_window_kv_max)
from .inputs import WORKLOADS, Workload, make_case, make_cell_map, to_cells
from .pipeline import SfaStep

__all__ = [n for n in dir() if not n.startswith("_")]

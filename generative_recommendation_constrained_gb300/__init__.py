"""GB300 (sm_103a) filtering-first constrained beam decoding over semantic IDs.

The product is the C-ABI library libzerogr.so (include/zerogr.h); this
package is its thin binding.  Importing it fails loudly if the library has
not been built (``__graft_entry__.build()``).
"""
from ._lib import (DTYPES, LIB_PATH, ZG_BF16, ZG_F16, ZG_F32, ZG_FMT_DENSE, ZG_FMT_SPARSE,
                   ZG_FORMAT_ALL_DENSE, ZG_FORMAT_ALL_SPARSE, ZG_FORMAT_AUTO, ZG_FULL, ZG_HIDDEN_SINGLE,
                   ZG_HIDDEN_SPLIT, ZG_INJECT_COPY, ZG_SCORES_AUTO, ZG_SCORES_CHUNK_TOPS, ZG_SCORES_WRITTEN,
                   ZG_INJECT_PINNED_ALLOC, ZG_NAIVE, ZG_MAX_BEAM, ZG_ORDER_FILTER_FIRST, ZG_ORDER_SCORE_FIRST,
                   ZG_RESIDENT_DEVICE, ZG_RESIDENT_HOST, ZG_SELECTIVE, ZG_STATIC_SCRATCH_BYTES, Index, Plan,
                   ZgError, make_model, zg_check_device_status, zg_debug_inject_build_failure,
                   zg_debug_set_wait_limit, zg_decode, zg_decode_host, zg_decode_host_workspace_size,
                   zg_decode_static, zg_decode_trace, zg_decode_workspace_size, zg_index_build,
                   zg_index_export, zg_index_info_get, zg_index_load, zg_index_save, zg_index_stats,
                   zg_plan_describe, zg_plan_force, zg_plan_load, zg_plan_save, zg_plan_set_fusion,
                   zg_plan_set_full_projection, zg_plan_set_order, zg_tune, zg_version)

__all__ = [
    "DTYPES", "LIB_PATH", "ZG_BF16", "ZG_F16", "ZG_F32", "ZG_FMT_DENSE", "ZG_FMT_SPARSE",
    "ZG_FORMAT_ALL_DENSE", "ZG_FORMAT_ALL_SPARSE", "ZG_FORMAT_AUTO", "ZG_FULL", "ZG_HIDDEN_SINGLE",
    "ZG_HIDDEN_SPLIT", "ZG_INJECT_COPY", "ZG_SCORES_AUTO", "ZG_SCORES_CHUNK_TOPS", "ZG_SCORES_WRITTEN",
    "ZG_INJECT_PINNED_ALLOC", "ZG_MAX_BEAM", "ZG_NAIVE", "ZG_ORDER_FILTER_FIRST", "ZG_ORDER_SCORE_FIRST",
    "ZG_RESIDENT_DEVICE", "ZG_RESIDENT_HOST", "ZG_SELECTIVE", "ZG_STATIC_SCRATCH_BYTES", "Index", "Plan",
    "ZgError", "make_model", "zg_check_device_status", "zg_debug_inject_build_failure",
    "zg_debug_set_wait_limit", "zg_decode", "zg_decode_host", "zg_decode_host_workspace_size",
    "zg_decode_static", "zg_decode_trace", "zg_decode_workspace_size", "zg_index_build",
    "zg_index_export", "zg_index_info_get", "zg_index_load", "zg_index_save", "zg_index_stats",
    "zg_plan_describe", "zg_plan_force", "zg_plan_load", "zg_plan_save", "zg_plan_set_fusion",
    "zg_plan_set_full_projection", "zg_plan_set_order", "zg_tune", "zg_version",
]

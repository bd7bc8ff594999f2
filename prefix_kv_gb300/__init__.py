"""Block-causal attention with a prefix K/V cache, native to NVIDIA GB300 (sm_103a).

The compute lives in ``lib/libbca_gb300.so`` (C ABI declared in ``include/bca.h``);
this package is its thin Python binding plus the seeded workload generator.
"""
from .api import (PagePool, check_status, new_status, pool_copy_rows,  # noqa: F401
                  prefix_cache_append_fp8_paged, prefix_cache_append_paged,
                  prefix_decode_fp8_paged, prefix_decode_paged, prefill, prefill_append,
                  prefill_piecewise,
                  prefill_piecewise_workspace_bytes, prefill_workspace_bytes,
                  prefix_cache_append, prefix_cache_append_fp8, prefix_decode, prefix_decode_fp8,
                  prefix_decode_fp8_workspace_bytes, prefix_decode_workspace_bytes,
                  prefix_cache_dequant_fp8,
                  qk_norm_rope_append, read_status, rope_positions, rope_table,
                  schedule_prep)

__all__ = ["prefill", "prefill_append", "prefix_decode", "prefix_decode_fp8", "prefix_decode_fp8_workspace_bytes",
           "prefix_cache_dequant_fp8", "prefix_cache_append", "prefix_cache_append_fp8", "schedule_prep",
           "prefill_workspace_bytes", "new_status", "read_status", "check_status",
           "rope_positions", "rope_table", "qk_norm_rope_append", "prefill_piecewise",
           "prefill_piecewise_workspace_bytes", "PagePool", "prefix_cache_append_paged",
           "prefix_decode_paged", "pool_copy_rows", "prefix_cache_append_fp8_paged",
           "prefix_decode_fp8_paged", "prefix_decode_workspace_bytes"]

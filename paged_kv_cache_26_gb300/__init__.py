"""GB300-native paged KV cache: slot-mapped KV append and single-token decode
attention over a block-table-addressed KV pool of fp16/bf16 values or E4M3
codes (hand-written sm_103a CUDA behind a C ABI), plus the host block allocator that produces the tables.

The shared library loads lazily on the first call; if it has not been built
every call raises (there is no fallback implementation)."""
from .api import (BlockAllocator, PagedKVError, make_workspace, paged_decode_attention,
                  paged_decode_attention_fp8, paged_decode_attention_no_alloc, paged_decode_step_fp8,
                  paged_kv_append_fp8, paged_decode_attention_multi, paged_decode_step_multi,
                  paged_decode_multi_workspace_bytes, paged_decode_multi_resolve_splits, paged_kv_slot_mapping_multi,
                  paged_kv_copy_blocks, paged_kv_selftest_wait, paged_kv_selftest_stale_prologue,
                  paged_decode_resolve_splits, paged_decode_step, paged_decode_step_from_host,
                  paged_decode_step_fp8_from_host, paged_decode_step_multi_from_host,
                  paged_decode_workspace_bytes,
                  paged_kv_append, paged_kv_check_status, paged_kv_slot_mapping)

__all__ = [
    "BlockAllocator", "PagedKVError", "make_workspace", "paged_decode_attention",
    "paged_decode_attention_no_alloc", "paged_decode_resolve_splits",
    "paged_decode_step", "paged_decode_step_from_host", "paged_decode_step_fp8_from_host",
    "paged_decode_step_multi_from_host",
    "paged_decode_workspace_bytes", "paged_kv_append",
    "paged_kv_check_status", "paged_kv_slot_mapping",
    "paged_kv_append_fp8", "paged_decode_attention_fp8", "paged_decode_step_fp8",
    "paged_decode_attention_multi", "paged_decode_step_multi", "paged_decode_multi_workspace_bytes",
    "paged_decode_multi_resolve_splits", "paged_kv_slot_mapping_multi", "paged_kv_copy_blocks",
    "paged_kv_selftest_wait", "paged_kv_selftest_stale_prologue",
]

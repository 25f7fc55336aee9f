"""ctypes loader for libpagedkv.so (built in-tree by build.py)."""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

c_int32_p = ctypes.POINTER(ctypes.c_int32)


class PkvDims(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int32) for name in (
        "num_seqs", "num_q_heads", "num_kv_heads", "head_dim", "block_size",
        "num_blocks", "max_blocks_per_seq", "dtype")]


class PkvStepBuffers(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in (
        "q_host", "k_new_host", "v_new_host", "block_tables_host", "context_lens_host", "out_host",
        "q_dev", "k_new_dev", "v_new_dev", "block_tables_dev", "context_lens_dev", "out_dev")]


class PkvEngineStats(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int64) for name in (
        "steps", "sequence_steps", "context_tokens", "unused_tail_slots", "copied_blocks")]


_SIGNATURES = {
    "paged_kv_append": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(PkvDims), ctypes.c_void_p]),
    "paged_decode_attention": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_int32,
                                              ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(PkvDims),
                                              ctypes.c_void_p]),
    "paged_decode_step": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
                                         ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t,
                                         ctypes.POINTER(PkvDims), ctypes.c_void_p]),
    "paged_decode_attention_no_alloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
                                                       ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(PkvDims),
                                                       ctypes.c_void_p]),
    "paged_decode_resolve_splits": (ctypes.c_int32, [ctypes.POINTER(PkvDims), ctypes.c_int32]),
    "paged_decode_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(PkvDims), ctypes.c_int32]),
    "paged_decode_step_from_host": (ctypes.c_int, [ctypes.POINTER(PkvStepBuffers), ctypes.c_void_p, ctypes.c_void_p,
                                                   ctypes.c_float, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t,
                                                   ctypes.POINTER(PkvDims), ctypes.c_void_p]),
    "paged_decode_step_multi_from_host": (ctypes.c_int, [ctypes.POINTER(PkvStepBuffers), ctypes.c_int32,
                                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
                                                         ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t,
                                                         ctypes.POINTER(PkvDims), ctypes.c_void_p]),
    "paged_decode_step_fp8_from_host": (ctypes.c_int, [ctypes.POINTER(PkvStepBuffers), ctypes.c_void_p,
                                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                       ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t,
                                                       ctypes.POINTER(PkvDims), ctypes.c_void_p]),
    "paged_kv_append_fp8": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                           ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.POINTER(PkvDims), ctypes.c_void_p]),
    "paged_decode_attention_fp8": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                  ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p,
                                                  ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(PkvDims),
                                                  ctypes.c_void_p]),
    "paged_decode_step_fp8": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_size_t, ctypes.POINTER(PkvDims), ctypes.c_void_p]),
    "paged_decode_attention_multi": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_float,
                                                    ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                                    ctypes.c_size_t, ctypes.POINTER(PkvDims), ctypes.c_void_p]),
    "paged_decode_step_multi": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                               ctypes.c_float, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                               ctypes.c_size_t, ctypes.POINTER(PkvDims), ctypes.c_void_p]),
    "paged_decode_step_multi_tc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                                  ctypes.c_float, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                                  ctypes.c_size_t, ctypes.POINTER(PkvDims), ctypes.c_void_p]),
    "paged_decode_multi_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(PkvDims), ctypes.c_int32,
                                                             ctypes.c_int32]),
    "paged_decode_multi_resolve_splits": (ctypes.c_int32, [ctypes.POINTER(PkvDims), ctypes.c_int32, ctypes.c_int32]),
    "paged_kv_slot_mapping_multi": (ctypes.c_int, [c_int32_p, c_int32_p, ctypes.c_int32, ctypes.c_int32,
                                                   ctypes.c_int32, ctypes.c_int32, c_int32_p]),
    "paged_kv_selftest_wait": (ctypes.c_int, [ctypes.c_void_p]),
    "paged_kv_selftest_stale_prologue": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                        ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                                                        ctypes.c_size_t, ctypes.c_int32, ctypes.POINTER(PkvDims),
                                                        ctypes.c_void_p]),
    "paged_kv_check_status": (ctypes.c_int, [ctypes.c_void_p]),
    "paged_kv_last_error": (ctypes.c_char_p, []),
    "paged_kv_slot_mapping": (ctypes.c_int, [c_int32_p, c_int32_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                             c_int32_p]),
    "block_allocator_create": (ctypes.c_void_p, [ctypes.c_int32, ctypes.c_int32, ctypes.c_uint64]),
    "block_allocator_destroy": (None, [ctypes.c_void_p]),
    "block_allocator_add_seq": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, c_int32_p]),
    "block_allocator_fork_prefix": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                   c_int32_p]),
    "block_allocator_append_slot": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, c_int32_p]),
    "block_allocator_append_slots": (ctypes.c_int, [ctypes.c_void_p, c_int32_p, ctypes.c_int32, c_int32_p]),
    "block_allocator_step_batch": (ctypes.c_int, [ctypes.c_void_p, c_int32_p, ctypes.c_int32, ctypes.c_int32,
                                                  c_int32_p, c_int32_p]),
    "block_allocator_free_seq": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    "block_allocator_fork": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, c_int32_p]),
    "block_allocator_append_slot_cow": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, c_int32_p, c_int32_p,
                                                       c_int32_p]),
    "block_allocator_step_batch_cow": (ctypes.c_int, [ctypes.c_void_p, c_int32_p, ctypes.c_int32, ctypes.c_int32,
                                                      c_int32_p, c_int32_p, c_int32_p, c_int32_p]),
    "paged_kv_copy_blocks": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                            ctypes.POINTER(PkvDims), ctypes.c_int32, ctypes.c_void_p]),
    "block_allocator_block_tables": (ctypes.c_int, [ctypes.c_void_p, c_int32_p, ctypes.c_int32, ctypes.c_int32,
                                                    c_int32_p, c_int32_p]),
    "block_allocator_num_free": (ctypes.c_int32, [ctypes.c_void_p]),
    "decode_engine_create": (ctypes.c_void_p, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32]),
    "decode_engine_destroy": (None, [ctypes.c_void_p]),
    "decode_engine_admit": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                           ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.POINTER(PkvDims), ctypes.c_void_p, c_int32_p]),
    "decode_engine_step": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(PkvDims),
                                          ctypes.c_void_p]),
    "decode_engine_last_step": (ctypes.c_int, [ctypes.c_void_p, c_int32_p, c_int32_p]),
    "decode_engine_get_stats": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(PkvEngineStats)]),
    "decode_engine_reset_stats": (ctypes.c_int, [ctypes.c_void_p]),
    "decode_engine_fork": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, c_int32_p]),
    "decode_engine_set_kv_scales": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "decode_engine_finish": (ctypes.c_int, [ctypes.c_void_p, c_int32_p, c_int32_p]),
    "decode_engine_state": (ctypes.c_int, [ctypes.c_void_p, c_int32_p, c_int32_p]),
    "block_allocator_refcount": (ctypes.c_int32, [ctypes.c_void_p, ctypes.c_int32]),
    "block_allocator_seq_len": (ctypes.c_int32, [ctypes.c_void_p, ctypes.c_int32]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built: there is no
    fallback implementation."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m paged_kv_cache_26_gb300.build` "
                "(nvcc, sm_103a); the paged KV path has no other implementation")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


EXPORTED = tuple(_SIGNATURES)

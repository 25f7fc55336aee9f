"""Python binding of libpagedkv.so: the same calls as the C ABI, taking torch
tensors.  Only argument marshalling happens here; every step of the decode
path runs in the library's CUDA kernels (or, for the allocator and slot
mapping, its host C++)."""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import numpy as np
import torch

from ._native import PkvDims, PkvStepBuffers, c_int32_p, lib

PKV_OK = 0
ERROR_NAMES = {
    -1: "PKV_ERR_INVALID_ARG", -2: "PKV_ERR_UNSUPPORTED", -3: "PKV_ERR_CUDA", -4: "PKV_ERR_TIMEOUT",
    -5: "PKV_ERR_NO_BLOCKS", -6: "PKV_ERR_OUT_OF_RANGE", -7: "PKV_ERR_SHARED_BLOCK",
}
_DTYPE_CODE = {torch.float16: 0, torch.bfloat16: 1}
STEP_KEYS = ("q", "k_new", "v_new", "block_tables", "context_lens", "out")


class PagedKVError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = lib().paged_kv_last_error().decode(errors="replace")
        super().__init__(f"{where}: {ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


def _check(code: int, where: str) -> int:
    if code < 0:
        raise PagedKVError(code, where)
    return code


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need_cuda(name: str, t: torch.Tensor, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def make_dims(q_or_new: torch.Tensor, k_cache: torch.Tensor, block_tables: Optional[torch.Tensor] = None,
              num_q_heads: Optional[int] = None) -> PkvDims:
    nb, hkv, bs, d = k_cache.shape
    if k_cache.dtype not in _DTYPE_CODE:
        raise ValueError("caches must be float16 or bfloat16")
    return PkvDims(num_seqs=q_or_new.shape[0],
                   num_q_heads=num_q_heads if num_q_heads is not None else q_or_new.shape[1],
                   num_kv_heads=hkv, head_dim=d, block_size=bs, num_blocks=nb,
                   max_blocks_per_seq=block_tables.shape[1] if block_tables is not None else 0,
                   dtype=_DTYPE_CODE[k_cache.dtype])


def _check_attention_shapes(q: torch.Tensor, out: torch.Tensor, k_cache: torch.Tensor,
                            block_tables: torch.Tensor, context_lens: torch.Tensor) -> None:
    """Shape checks shared by the one-token attention calls, made before any
    launch: the kernels read context_lens[b] and row b of block_tables for
    every sequence b of q, so both must have a row per sequence."""
    if out.shape != q.shape or q.dim() != 3 or q.shape[2] != k_cache.shape[3]:
        raise ValueError("q / out must be [num_seqs][num_q_heads][head_dim]")
    if block_tables.dim() != 2 or block_tables.shape[0] != q.shape[0] or context_lens.shape != (q.shape[0],):
        raise ValueError("block_tables must be [num_seqs][max_blocks], context_lens [num_seqs]")


def paged_kv_append(k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                    k_cache: torch.Tensor, v_cache: torch.Tensor, stream=None) -> None:
    """Store token i's K/V (k_new[i], v_new[i]: [Hkv][D]) at slot slot_mapping[i]
    of the paged caches ([NB][Hkv][16][D]); negative slots are skipped."""
    for n, t in (("k_new", k_new), ("v_new", v_new), ("k_cache", k_cache), ("v_cache", v_cache)):
        _need_cuda(n, t, k_cache.dtype)
    _need_cuda("slot_mapping", slot_mapping, torch.int32)
    if k_new.shape != v_new.shape or k_new.shape[1:] != (k_cache.shape[1], k_cache.shape[3]):
        raise ValueError("k_new / v_new must be [num_tokens][num_kv_heads][head_dim] matching the cache")
    if k_cache.shape != v_cache.shape or slot_mapping.shape != (k_new.shape[0],):
        raise ValueError("cache shapes differ or slot_mapping is not [num_tokens]")
    dims = make_dims(k_new, k_cache, num_q_heads=k_cache.shape[1])
    _check(lib().paged_kv_append(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), k_new.shape[0],
                                 _ptr(k_cache), _ptr(v_cache), ctypes.byref(dims), _stream(stream)),
           "paged_kv_append")


def paged_decode_resolve_splits(q: torch.Tensor, k_cache: torch.Tensor, block_tables: torch.Tensor,
                                num_splits: int = 0) -> int:
    dims = make_dims(q, k_cache, block_tables)
    return _check(lib().paged_decode_resolve_splits(ctypes.byref(dims), num_splits), "paged_decode_resolve_splits")


def paged_decode_workspace_bytes(q: torch.Tensor, k_cache: torch.Tensor, block_tables: torch.Tensor,
                                 num_splits: int = 0) -> int:
    dims = make_dims(q, k_cache, block_tables)
    return int(lib().paged_decode_workspace_bytes(ctypes.byref(dims), num_splits))


def make_workspace(q: torch.Tensor, k_cache: torch.Tensor, block_tables: torch.Tensor,
                   num_splits: int = 0) -> Optional[torch.Tensor]:
    """A zero-filled workspace of the size paged_decode_attention needs (None if none)."""
    need = paged_decode_workspace_bytes(q, k_cache, block_tables, num_splits)
    return torch.zeros(need, dtype=torch.uint8, device=q.device) if need else None


def paged_decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                           out: Optional[torch.Tensor] = None, num_splits: int = 0,
                           workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out[b][h] = softmax(scale * q[b][h] K^T) V over the first context_lens[b]
    tokens of sequence b, K/V read through block_tables.  Returns out."""
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _need_cuda(n, t, k_cache.dtype)
    _need_cuda("block_tables", block_tables, torch.int32)
    _need_cuda("context_lens", context_lens, torch.int32)
    if out is None:
        out = torch.empty_like(q)
    _need_cuda("out", out, q.dtype)
    _check_attention_shapes(q, out, k_cache, block_tables, context_lens)
    dims = make_dims(q, k_cache, block_tables)
    need = int(lib().paged_decode_workspace_bytes(ctypes.byref(dims), num_splits))
    if need and workspace is None:
        # Caller did not supply one: allocate through torch (the library itself
        # never allocates).  Zero-filled: the kernels expect zeroed counters.
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().paged_decode_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                        _ptr(context_lens), float(scale), _ptr(out), num_splits,
                                        _ptr(workspace), ws_bytes, ctypes.byref(dims), _stream(stream)),
           "paged_decode_attention")
    return out


def paged_decode_attention_no_alloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                    block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                                    out: torch.Tensor, num_splits: int = 0, stream=None) -> torch.Tensor:
    """paged_decode_attention for callers that cannot allocate device memory
    while they run (plugin hosts that forbid it, processes whose memory another
    allocator holds, latency paths that cannot take cudaMalloc's
    synchronisation): the split scratch is a fixed 16 MiB array inside the
    library, so neither this wrapper nor the library allocates; ``out`` must be
    supplied.  Calls that overlap on the GPU share that array and race."""
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("out", out)):
        _need_cuda(n, t, k_cache.dtype)
    _need_cuda("block_tables", block_tables, torch.int32)
    _need_cuda("context_lens", context_lens, torch.int32)
    _check_attention_shapes(q, out, k_cache, block_tables, context_lens)
    dims = make_dims(q, k_cache, block_tables)
    _check(lib().paged_decode_attention_no_alloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                                 _ptr(context_lens), float(scale), _ptr(out), num_splits,
                                                 ctypes.byref(dims), _stream(stream)),
           "paged_decode_attention_no_alloc")
    return out


def paged_decode_step(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                      out: Optional[torch.Tensor] = None, num_splits: int = 0,
                      workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """One decode step: store each sequence's new token (k_new[b], v_new[b])
    at position context_lens[b] - 1 through its block table, then attend over
    positions [0, context_lens[b]).  Returns out."""
    for n, t in (("q", q), ("k_new", k_new), ("v_new", v_new), ("k_cache", k_cache), ("v_cache", v_cache)):
        _need_cuda(n, t, k_cache.dtype)
    _need_cuda("block_tables", block_tables, torch.int32)
    _need_cuda("context_lens", context_lens, torch.int32)
    if out is None:
        out = torch.empty_like(q)
    _need_cuda("out", out, q.dtype)
    if k_new.shape != (q.shape[0], k_cache.shape[1], k_cache.shape[3]) or v_new.shape != k_new.shape:
        raise ValueError("k_new / v_new must be [num_seqs][num_kv_heads][head_dim]")
    _check_attention_shapes(q, out, k_cache, block_tables, context_lens)
    dims = make_dims(q, k_cache, block_tables)
    need = int(lib().paged_decode_workspace_bytes(ctypes.byref(dims), num_splits))
    if need and workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().paged_decode_step(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(block_tables), _ptr(context_lens), float(scale), _ptr(out), num_splits,
                                   _ptr(workspace), ws_bytes, ctypes.byref(dims), _stream(stream)),
           "paged_decode_step")
    return out


def paged_decode_step_from_host(host: dict, dev: dict, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                scale: float, num_splits: int = 0, workspace: Optional[torch.Tensor] = None,
                                stream=None) -> None:
    """One decode step from (pinned) host buffers: copies q, k_new, v_new,
    block_tables, context_lens into the device staging tensors in ``dev``,
    runs paged_decode_step, and copies out back into host['out'].
    Keys of both dicts: q, k_new, v_new, block_tables, context_lens, out."""
    keys = STEP_KEYS
    bufs = PkvStepBuffers(**{f"{k}_host": host[k].data_ptr() for k in keys},
                          **{f"{k}_dev": dev[k].data_ptr() for k in keys})
    dims = make_dims(dev["q"], k_cache, dev["block_tables"])
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().paged_decode_step_from_host(ctypes.byref(bufs), _ptr(k_cache), _ptr(v_cache), float(scale),
                                             num_splits, _ptr(workspace), ws_bytes, ctypes.byref(dims),
                                             _stream(stream)),
           "paged_decode_step_from_host")


def paged_decode_step_fp8_from_host(host: dict, dev: dict, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                    k_scale: torch.Tensor, v_scale: torch.Tensor, scale: float,
                                    workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """paged_decode_step_from_host over E4M3 pools (uint8 codes with float32
    per-KV-head scales k_scale / v_scale); q / k_new / v_new / out stay fp16 or
    bf16.  Same dict keys as paged_decode_step_from_host."""
    for n, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        _need_cuda(n, t, torch.float32)
    keys = STEP_KEYS
    bufs = PkvStepBuffers(**{f"{k}_host": host[k].data_ptr() for k in keys},
                          **{f"{k}_dev": dev[k].data_ptr() for k in keys})
    dims = make_dims_fp8(dev["q"], k_cache, dev["block_tables"])
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().paged_decode_step_fp8_from_host(ctypes.byref(bufs), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                                 _ptr(v_scale), float(scale), _ptr(workspace), ws_bytes,
                                                 ctypes.byref(dims), _stream(stream)),
           "paged_decode_step_fp8_from_host")


# ---------------------------------------------------------------- several new tokens per sequence

def _multi_checks(q, k_cache, v_cache, block_tables, context_lens, out):
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _need_cuda(n, t, k_cache.dtype)
    _need_cuda("block_tables", block_tables, torch.int32)
    _need_cuda("context_lens", context_lens, torch.int32)
    _need_cuda("out", out, q.dtype)
    if q.dim() != 4 or out.shape != q.shape or q.shape[3] != k_cache.shape[3] or k_cache.shape != v_cache.shape:
        raise ValueError("q / out must be [num_seqs][q_len][num_q_heads][head_dim] matching the caches")
    if block_tables.dim() != 2 or block_tables.shape[0] != q.shape[0] or context_lens.shape != (q.shape[0],):
        raise ValueError("block_tables must be [num_seqs][max_blocks], context_lens [num_seqs]")


def _multi_dims(q, k_cache, block_tables):
    return make_dims(q, k_cache, block_tables, num_q_heads=q.shape[2])


def paged_decode_multi_workspace_bytes(q: torch.Tensor, k_cache: torch.Tensor, block_tables: torch.Tensor,
                                       num_splits: int = 0) -> int:
    dims = _multi_dims(q, k_cache, block_tables)
    return int(lib().paged_decode_multi_workspace_bytes(ctypes.byref(dims), q.shape[1], num_splits))


def paged_decode_multi_resolve_splits(q: torch.Tensor, k_cache: torch.Tensor, block_tables: torch.Tensor,
                                      num_splits: int = 0) -> int:
    dims = _multi_dims(q, k_cache, block_tables)
    return _check(lib().paged_decode_multi_resolve_splits(ctypes.byref(dims), q.shape[1], num_splits),
                  "paged_decode_multi_resolve_splits")


def _multi_workspace(q, k_cache, block_tables, num_splits, workspace):
    need = paged_decode_multi_workspace_bytes(q, k_cache, block_tables, num_splits)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    return workspace, (workspace.numel() * workspace.element_size() if workspace is not None else 0)


def paged_decode_attention_multi(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                 block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                                 out: Optional[torch.Tensor] = None, num_splits: int = 0,
                                 workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode attention for q.shape[1] new tokens per sequence (q:
    [B][q_len][Hq][D]): new token i of sequence b, at position
    context_lens[b] - q_len + i, attends to positions 0 .. itself."""
    if out is None:
        out = torch.empty_like(q)
    _multi_checks(q, k_cache, v_cache, block_tables, context_lens, out)
    dims = _multi_dims(q, k_cache, block_tables)
    workspace, ws_bytes = _multi_workspace(q, k_cache, block_tables, num_splits, workspace)
    _check(lib().paged_decode_attention_multi(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                              _ptr(context_lens), q.shape[1], float(scale), _ptr(out), num_splits,
                                              _ptr(workspace), ws_bytes, ctypes.byref(dims), _stream(stream)),
           "paged_decode_attention_multi")
    return out


def paged_decode_step_multi(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                            v_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                            scale: float, out: Optional[torch.Tensor] = None, num_splits: int = 0,
                            workspace: Optional[torch.Tensor] = None, stream=None,
                            tensor_cores: bool = False) -> torch.Tensor:
    """Append the q_len new tokens' K/V (k_new, v_new: [B][q_len][Hkv][D]) at
    positions context_lens[b] - q_len .. context_lens[b] - 1, then
    paged_decode_attention_multi.  tensor_cores: run the tcgen05 kernel
    (paged_decode_step_multi_tc; 64 query rows per KV head only)."""
    if out is None:
        out = torch.empty_like(q)
    _multi_checks(q, k_cache, v_cache, block_tables, context_lens, out)
    for n, t in (("k_new", k_new), ("v_new", v_new)):
        _need_cuda(n, t, k_cache.dtype)
    if k_new.shape != (q.shape[0], q.shape[1], k_cache.shape[1], k_cache.shape[3]) or v_new.shape != k_new.shape:
        raise ValueError("k_new / v_new must be [num_seqs][q_len][num_kv_heads][head_dim]")
    dims = _multi_dims(q, k_cache, block_tables)
    workspace, ws_bytes = _multi_workspace(q, k_cache, block_tables, num_splits, workspace)
    name = "paged_decode_step_multi_tc" if tensor_cores else "paged_decode_step_multi"
    _check(getattr(lib(), name)(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                _ptr(block_tables), _ptr(context_lens), q.shape[1], float(scale), _ptr(out),
                                num_splits, _ptr(workspace), ws_bytes, ctypes.byref(dims), _stream(stream)),
           name)
    return out


def paged_decode_step_multi_from_host(host: dict, dev: dict, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                      scale: float, num_splits: int = 0, workspace: Optional[torch.Tensor] = None,
                                      stream=None) -> None:
    """paged_decode_step_multi from (pinned) host buffers: q / k_new / v_new /
    out hold q_len rows per sequence ([B][q_len][...]); same dict keys as
    paged_decode_step_from_host.  A workspace is allocated when the call needs
    one and none is given."""
    keys = STEP_KEYS
    q_len = int(dev["q"].shape[1])
    bufs = PkvStepBuffers(**{f"{k}_host": host[k].data_ptr() for k in keys},
                          **{f"{k}_dev": dev[k].data_ptr() for k in keys})
    dims = _multi_dims(dev["q"], k_cache, dev["block_tables"])
    workspace, ws_bytes = _multi_workspace(dev["q"], k_cache, dev["block_tables"], num_splits, workspace)
    _check(lib().paged_decode_step_multi_from_host(ctypes.byref(bufs), q_len, _ptr(k_cache), _ptr(v_cache),
                                                   float(scale), num_splits, _ptr(workspace), ws_bytes,
                                                   ctypes.byref(dims), _stream(stream)),
           "paged_decode_step_multi_from_host")


def paged_kv_slot_mapping_multi(block_tables: np.ndarray, context_lens: np.ndarray, q_len: int,
                                block_size: int = 16) -> np.ndarray:
    """Host: slots [B][q_len] of each sequence's q_len newest tokens (-1 below position 0)."""
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.empty((cl.shape[0], q_len), dtype=np.int32)
    _check(lib().paged_kv_slot_mapping_multi(bt.ctypes.data_as(c_int32_p), cl.ctypes.data_as(c_int32_p),
                                             cl.shape[0], bt.shape[1] if bt.ndim == 2 else 0, block_size, q_len,
                                             out.ctypes.data_as(c_int32_p)),
           "paged_kv_slot_mapping_multi")
    return out


# ---------------------------------------------------------------- FP8 (E4M3) cache

_FP8_CACHE_DTYPES = (torch.uint8, torch.float8_e4m3fn)


def _need_fp8_cache(name: str, t: torch.Tensor):
    _need_cuda(name, t)
    if t.dtype not in _FP8_CACHE_DTYPES:
        raise ValueError(f"{name} must hold E4M3 codes (uint8 or float8_e4m3fn), got {t.dtype}")


def _need_scales(k_scale: torch.Tensor, v_scale: torch.Tensor, hkv: int):
    for n, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        _need_cuda(n, t, torch.float32)
        if t.shape != (hkv,):
            raise ValueError(f"{n} must be float32[num_kv_heads]")


def make_dims_fp8(q_or_new: torch.Tensor, k_cache: torch.Tensor, block_tables: Optional[torch.Tensor] = None,
                  num_q_heads: Optional[int] = None) -> PkvDims:
    """Dims of a call over an E4M3 pool: dtype is that of q / out / k_new / v_new."""
    nb, hkv, bs, d = k_cache.shape
    if q_or_new.dtype not in _DTYPE_CODE:
        raise ValueError("q / k_new / v_new must be float16 or bfloat16")
    return PkvDims(num_seqs=q_or_new.shape[0],
                   num_q_heads=num_q_heads if num_q_heads is not None else q_or_new.shape[1],
                   num_kv_heads=hkv, head_dim=d, block_size=bs, num_blocks=nb,
                   max_blocks_per_seq=block_tables.shape[1] if block_tables is not None else 0,
                   dtype=_DTYPE_CODE[q_or_new.dtype])


def paged_kv_append_fp8(k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                        k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: torch.Tensor,
                        v_scale: torch.Tensor, stream=None) -> None:
    """paged_kv_append into E4M3 caches: token i's K/V of KV head h are stored
    as E4M3(x / k_scale[h]) and E4M3(x / v_scale[h])."""
    _need_cuda("k_new", k_new)
    _need_cuda("v_new", v_new, k_new.dtype)
    _need_cuda("slot_mapping", slot_mapping, torch.int32)
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _need_fp8_cache(n, t)
    _need_scales(k_scale, v_scale, k_cache.shape[1])
    if k_new.shape != v_new.shape or k_new.shape[1:] != (k_cache.shape[1], k_cache.shape[3]):
        raise ValueError("k_new / v_new must be [num_tokens][num_kv_heads][head_dim] matching the cache")
    if k_cache.shape != v_cache.shape or slot_mapping.shape != (k_new.shape[0],):
        raise ValueError("cache shapes differ or slot_mapping is not [num_tokens]")
    dims = make_dims_fp8(k_new, k_cache, num_q_heads=k_cache.shape[1])
    _check(lib().paged_kv_append_fp8(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), k_new.shape[0], _ptr(k_cache),
                                     _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), ctypes.byref(dims),
                                     _stream(stream)),
           "paged_kv_append_fp8")


def _fp8_call_checks(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, out):
    _need_cuda("q", q)
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _need_fp8_cache(n, t)
    _need_scales(k_scale, v_scale, k_cache.shape[1])
    _need_cuda("block_tables", block_tables, torch.int32)
    _need_cuda("context_lens", context_lens, torch.int32)
    _need_cuda("out", out, q.dtype)
    if out.shape != q.shape or q.dim() != 3 or q.shape[2] != k_cache.shape[3] or k_cache.shape != v_cache.shape:
        raise ValueError("q / out must be [num_seqs][num_q_heads][head_dim] matching the caches")
    if block_tables.dim() != 2 or block_tables.shape[0] != q.shape[0] or context_lens.shape != (q.shape[0],):
        raise ValueError("block_tables must be [num_seqs][max_blocks], context_lens [num_seqs]")


def _fp8_workspace(dims, q, workspace):
    need = int(lib().paged_decode_workspace_bytes(ctypes.byref(dims), 0))
    if need and workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return workspace, ws_bytes


def paged_decode_attention_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                               k_scale: torch.Tensor, v_scale: torch.Tensor, block_tables: torch.Tensor,
                               context_lens: torch.Tensor, scale: float, out: Optional[torch.Tensor] = None,
                               workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """paged_decode_attention over E4M3 caches with per-KV-head scales."""
    if out is None:
        out = torch.empty_like(q)
    _fp8_call_checks(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, out)
    dims = make_dims_fp8(q, k_cache, block_tables)
    workspace, ws_bytes = _fp8_workspace(dims, q, workspace)
    _check(lib().paged_decode_attention_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                            _ptr(block_tables), _ptr(context_lens), float(scale), _ptr(out),
                                            _ptr(workspace), ws_bytes, ctypes.byref(dims), _stream(stream)),
           "paged_decode_attention_fp8")
    return out


def paged_decode_step_fp8(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                          v_cache: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor,
                          block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                          out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
    """paged_decode_step over E4M3 caches: the new token is quantised with
    the scales and appended, then attended, in one fused launch."""
    if out is None:
        out = torch.empty_like(q)
    _fp8_call_checks(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, out)
    _need_cuda("k_new", k_new, q.dtype)
    _need_cuda("v_new", v_new, q.dtype)
    if k_new.shape != (q.shape[0], k_cache.shape[1], k_cache.shape[3]) or v_new.shape != k_new.shape:
        raise ValueError("k_new / v_new must be [num_seqs][num_kv_heads][head_dim]")
    dims = make_dims_fp8(q, k_cache, block_tables)
    workspace, ws_bytes = _fp8_workspace(dims, q, workspace)
    _check(lib().paged_decode_step_fp8(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                       _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), _ptr(context_lens),
                                       float(scale), _ptr(out), _ptr(workspace), ws_bytes, ctypes.byref(dims),
                                       _stream(stream)),
           "paged_decode_step_fp8")
    return out


def paged_kv_copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, block_pairs: torch.Tensor,
                         stream=None) -> None:
    """Copy-on-write: for each row (src, dst) of block_pairs (int32 [n][2] on
    the device), physical block dst of both caches becomes a copy of block src.
    Caches: fp16/bf16 [NB][Hkv][16][D] or E4M3 codes (uint8 / float8_e4m3fn)."""
    _need_cuda("k_cache", k_cache)
    _need_cuda("v_cache", v_cache, k_cache.dtype)
    _need_cuda("block_pairs", block_pairs, torch.int32)
    if block_pairs.dim() != 2 or block_pairs.shape[1] != 2:
        raise ValueError("block_pairs must be int32 [n][2]")
    if k_cache.shape != v_cache.shape or k_cache.dim() != 4:
        raise ValueError("caches must both be [num_blocks][num_kv_heads][16][head_dim]")
    nb, hkv, bs, d = k_cache.shape
    dims = PkvDims(num_seqs=0, num_q_heads=hkv, num_kv_heads=hkv, head_dim=d, block_size=bs, num_blocks=nb,
                   max_blocks_per_seq=0, dtype=_DTYPE_CODE.get(k_cache.dtype, 0))
    _check(lib().paged_kv_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(block_pairs), block_pairs.shape[0],
                                      ctypes.byref(dims), k_cache.element_size(), _stream(stream)),
           "paged_kv_copy_blocks")


def paged_kv_selftest_wait(stream=None) -> None:
    """Launch the bounded-wait self-test: the next paged_kv_check_status
    raises PagedKVError with PKV_ERR_TIMEOUT (-4) after about 1.5 s."""
    _check(lib().paged_kv_selftest_wait(_stream(stream)), "paged_kv_selftest_wait")


def paged_kv_selftest_stale_prologue(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                                     k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                                     context_lens: torch.Tensor, stale_block_tables: torch.Tensor,
                                     stale_context_lens: torch.Tensor, scale: float,
                                     out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                                     stream=None, publish: bool = True) -> torch.Tensor:
    """paged_decode_step (automatic path) whose kernels read the stale
    tables / lengths before their grid wait, as if the real ones were still
    being written: the result must be that of the real inputs.  With publish
    False the decode grid does not hand its validated lengths to the merge
    (as under stream capture), so the merge rebuilds its own plan after its
    wait.  Returns out."""
    for n, t in (("q", q), ("k_new", k_new), ("v_new", v_new), ("k_cache", k_cache), ("v_cache", v_cache)):
        _need_cuda(n, t, k_cache.dtype)
    for n, t in (("block_tables", block_tables), ("context_lens", context_lens),
                 ("stale_block_tables", stale_block_tables), ("stale_context_lens", stale_context_lens)):
        _need_cuda(n, t, torch.int32)
    if out is None:
        out = torch.empty_like(q)
    _need_cuda("out", out, q.dtype)
    _check_attention_shapes(q, out, k_cache, block_tables, context_lens)
    if stale_block_tables.shape != block_tables.shape or stale_context_lens.shape != context_lens.shape:
        raise ValueError("stale inputs must have the shapes of the real ones")
    if k_new.shape != (q.shape[0], k_cache.shape[1], k_cache.shape[3]) or v_new.shape != k_new.shape:
        raise ValueError("k_new / v_new must be [num_seqs][num_kv_heads][head_dim]")
    dims = make_dims(q, k_cache, block_tables)
    need = int(lib().paged_decode_workspace_bytes(ctypes.byref(dims), 0))
    if need and workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().paged_kv_selftest_stale_prologue(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        _ptr(stale_block_tables), _ptr(stale_context_lens), float(scale), _ptr(out), _ptr(workspace), ws_bytes,
        1 if publish else 0, ctypes.byref(dims), _stream(stream)), "paged_kv_selftest_stale_prologue")
    return out


def paged_kv_check_status(stream=None) -> None:
    """Synchronise the stream and raise if a kernel flagged an error."""
    _check(lib().paged_kv_check_status(_stream(stream)), "paged_kv_check_status")


def paged_kv_slot_mapping(block_tables: np.ndarray, context_lens: np.ndarray, block_size: int = 16) -> np.ndarray:
    """Host: slot of each sequence's newest token (position context_len - 1)."""
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.empty(cl.shape[0], dtype=np.int32)
    _check(lib().paged_kv_slot_mapping(bt.ctypes.data_as(c_int32_p), cl.ctypes.data_as(c_int32_p), cl.shape[0],
                                       bt.shape[1] if bt.ndim == 2 else 0, block_size,
                                       out.ctypes.data_as(c_int32_p)),
           "paged_kv_slot_mapping")
    return out


class BlockAllocator:
    """Host block pool: seeded scattered placement, reference counts, shared
    prefixes and per-token growth (the C++ allocator behind the C ABI)."""

    def __init__(self, num_blocks: int, block_size: int = 16, seed: int = 0):
        self._h = lib().block_allocator_create(num_blocks, block_size, seed)
        if not self._h:
            raise PagedKVError(-1, "block_allocator_create")
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self):
        if self._h:
            lib().block_allocator_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_seq(self, num_tokens: int) -> int:
        sid = ctypes.c_int32()
        _check(lib().block_allocator_add_seq(self._h, num_tokens, ctypes.byref(sid)), "add_seq")
        return sid.value

    def fork_prefix(self, src_seq: int, prefix_tokens: int, num_tokens: int) -> int:
        sid = ctypes.c_int32()
        _check(lib().block_allocator_fork_prefix(self._h, src_seq, prefix_tokens, num_tokens, ctypes.byref(sid)),
               "fork_prefix")
        return sid.value

    def append_slot(self, seq_id: int) -> int:
        slot = ctypes.c_int32()
        _check(lib().block_allocator_append_slot(self._h, seq_id, ctypes.byref(slot)), "append_slot")
        return slot.value

    def append_slots(self, seq_ids: Sequence[int], out: Optional[np.ndarray] = None) -> np.ndarray:
        """One new token for each listed sequence (all or nothing); returns the slots."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
        slots = out if out is not None else np.empty(ids.shape[0], dtype=np.int32)
        _check(lib().block_allocator_append_slots(self._h, ids.ctypes.data_as(c_int32_p), ids.shape[0],
                                                  slots.ctypes.data_as(c_int32_p)), "append_slots")
        return slots

    def step_batch(self, slot_seq_ids: np.ndarray, max_blocks: int, tables: np.ndarray, lens: np.ndarray) -> None:
        """Grow every live sequence of the batch by one token and write all
        rows of ``tables`` / ``lens`` (int32, C-contiguous, filled in place)."""
        ids = np.ascontiguousarray(slot_seq_ids, dtype=np.int32)
        _check(lib().block_allocator_step_batch(self._h, ids.ctypes.data_as(c_int32_p), ids.shape[0], max_blocks,
                                                tables.ctypes.data_as(c_int32_p), lens.ctypes.data_as(c_int32_p)),
               "step_batch")

    def fork(self, src_seq: int, prefix_tokens: int) -> int:
        """A new sequence sharing the blocks of src_seq's first prefix_tokens
        tokens (any count; the last shared block may be partly filled)."""
        sid = ctypes.c_int32()
        _check(lib().block_allocator_fork(self._h, src_seq, prefix_tokens, ctypes.byref(sid)), "fork")
        return sid.value

    def append_slot_cow(self, seq_id: int):
        """Grow seq_id by one token, copying a shared block first: returns
        (slot, copy) with copy = (src, dst) or None."""
        slot, n = ctypes.c_int32(), ctypes.c_int32()
        pair = (ctypes.c_int32 * 2)()
        _check(lib().block_allocator_append_slot_cow(self._h, seq_id, ctypes.byref(slot), pair, ctypes.byref(n)),
               "append_slot_cow")
        return slot.value, ((pair[0], pair[1]) if n.value else None)

    def step_batch_cow(self, slot_seq_ids: np.ndarray, max_blocks: int, tables: np.ndarray, lens: np.ndarray,
                       copy_pairs: np.ndarray) -> int:
        """step_batch with copy-on-write; copy_pairs (int32 [n][2], filled in
        place) receives the block copies to perform first.  Returns their count."""
        ids = np.ascontiguousarray(slot_seq_ids, dtype=np.int32)
        n = ctypes.c_int32()
        _check(lib().block_allocator_step_batch_cow(self._h, ids.ctypes.data_as(c_int32_p), ids.shape[0], max_blocks,
                                                    tables.ctypes.data_as(c_int32_p), lens.ctypes.data_as(c_int32_p),
                                                    copy_pairs.ctypes.data_as(c_int32_p), ctypes.byref(n)),
               "step_batch_cow")
        return n.value

    def free_seq(self, seq_id: int) -> None:
        _check(lib().block_allocator_free_seq(self._h, seq_id), "free_seq")

    def block_tables(self, seq_ids: Sequence[int], max_blocks: int):
        ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
        tables = np.empty((ids.shape[0], max_blocks), dtype=np.int32)
        lens = np.empty(ids.shape[0], dtype=np.int32)
        _check(lib().block_allocator_block_tables(self._h, ids.ctypes.data_as(c_int32_p), ids.shape[0], max_blocks,
                                                  tables.ctypes.data_as(c_int32_p), lens.ctypes.data_as(c_int32_p)),
               "block_tables")
        return tables, lens

    @property
    def num_free(self) -> int:
        return int(lib().block_allocator_num_free(self._h))

    def refcount(self, block: int) -> int:
        return int(lib().block_allocator_refcount(self._h, block))

    def seq_len(self, seq_id: int) -> int:
        return int(lib().block_allocator_seq_len(self._h, seq_id))

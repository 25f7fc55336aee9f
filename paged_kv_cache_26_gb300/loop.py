"""Continuous batching over the paged KV cache (Python face of the native
decode engine in the library).

A decode loop with a fixed number of batch slots, after the lifecycle the
pages describe (kasblo.com "vLLMとは？", section "blockはrequestの成長に合わせて
割り当てる": take blocks for the prompt, add one when the current block fills,
return a request's blocks when it ends so later requests reuse them; magi
"Inference Batching", continuous batching: finished sequences leave and
waiting ones enter at every iteration):

* admit(): a new sequence takes a free batch slot and the blocks its prompt
  needs; the prompt's K/V (produced elsewhere: prefill is not this path) is
  written through a slot-mapped append;
* step(): every active sequence gets one token: the engine grows each
  sequence (a new block at a block boundary), writes the block tables into
  mapped pinned host memory that the kernels read in place (no copy) and runs
  one paged_decode_step (append + attention) -- one native call per step;
* fork(): parallel sampling -- a new sequence sharing all of an active one's
  blocks; the shared block a step writes into is copied first (copy-on-write,
  kasblo.com "vLLMとは？", section "block共有とAutomatic Prefix Caching");
* finish_step(): sequences whose generation budget is spent free their blocks.

Empty batch slots have context length 0 (zero output, nothing appended).

With ``k_scale`` / ``v_scale`` (float32[num_kv_heads]) the pools hold E4M3
codes (design.babushkai.com "GPU推論の内部構造", section "KVキャッシュの台帳":
an FP8 cache halves the bytes per token); prompts and new tokens stay
fp16/bf16 and are quantised as they are appended.
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional

import numpy as np
import torch

from . import api
from ._native import PkvEngineStats, c_int32_p, lib

BLOCK_SIZE = 16


class DecodeLoop:
    def __init__(self, num_blocks: int, num_q_heads: int, num_kv_heads: int, head_dim: int, max_batch: int,
                 max_context: int, dtype=torch.bfloat16, device="cuda", seed: int = 0,
                 k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None):
        self.device = torch.device(device)
        self.dtype = dtype
        self.H, self.Hk, self.D = num_q_heads, num_kv_heads, head_dim
        self.B = max_batch
        self.max_blocks = math.ceil(max_context / BLOCK_SIZE)
        self.fp8 = k_scale is not None
        if self.fp8 != (v_scale is not None):
            raise ValueError("give both k_scale and v_scale, or neither")
        cache_dtype = torch.uint8 if self.fp8 else dtype
        self.k_cache = torch.zeros(num_blocks, num_kv_heads, BLOCK_SIZE, head_dim, dtype=cache_dtype,
                                   device=self.device)
        self.v_cache = torch.zeros_like(self.k_cache)
        if self.fp8:
            for n, t in (("k_scale", k_scale), ("v_scale", v_scale)):
                api._need_cuda(n, t, torch.float32)
                if t.shape != (num_kv_heads,):
                    raise ValueError(f"{n} must be float32[num_kv_heads]")
            self.k_scale, self.v_scale = k_scale, v_scale
        self.alloc = api.BlockAllocator(num_blocks, BLOCK_SIZE, seed)
        self._eng = lib().decode_engine_create(self.alloc._h, max_batch, self.max_blocks)
        if not self._eng:
            raise api.PagedKVError(-3, "decode_engine_create")
        self.out = torch.empty(max_batch, num_q_heads, head_dim, dtype=dtype, device=self.device)
        probe_q = torch.empty(max_batch, num_q_heads, head_dim, dtype=dtype, device=self.device)
        if self.fp8:
            api._check(lib().decode_engine_set_kv_scales(self._eng, ctypes.c_void_p(k_scale.data_ptr()),
                                                         ctypes.c_void_p(v_scale.data_ptr())), "set_kv_scales")
            self._dims = api.make_dims_fp8(probe_q, self.k_cache)
        else:
            self._dims = api.make_dims(probe_q, self.k_cache)
        self._dims.max_blocks_per_seq = self.max_blocks
        need = int(lib().paged_decode_workspace_bytes(ctypes.byref(self._dims), 0))
        self.workspace = torch.zeros(need, dtype=torch.uint8, device=self.device) if need else None
        self._freed = np.empty(max_batch, np.int32)
        self._nfreed = ctypes.c_int32(0)
        self._slot = ctypes.c_int32(-1)
        self._seq = np.full(max_batch, -1, np.int32)
        self._lens = np.zeros(max_batch, np.int32)
        self._step_args = None
        self._step_key = None
        self._num_free = max_batch
        self.steps = 0

    def close(self):
        if getattr(self, "_eng", None):
            lib().decode_engine_destroy(self._eng)
            self._eng = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------------ lifecycle

    def _state(self):
        api._check(lib().decode_engine_state(self._eng, self._seq.ctypes.data_as(c_int32_p),
                                             self._lens.ctypes.data_as(c_int32_p)), "decode_engine_state")

    @property
    def seq(self) -> np.ndarray:
        """Sequence id of every batch slot (-1 = empty)."""
        self._state()
        return self._seq.copy()

    def free_slots(self):
        return np.flatnonzero(self.seq < 0)

    @property
    def num_free_slots(self) -> int:
        """Empty batch slots (kept on the host side of the binding: no native call)."""
        return self._num_free

    def active_slots(self):
        return np.flatnonzero(self.seq >= 0)

    def admit(self, prompt_k: torch.Tensor, prompt_v: torch.Tensor, gen_len: int) -> Optional[int]:
        """Start a sequence whose prompt K/V are prompt_k / prompt_v
        ([P][Hkv][D] on the device); it will run for gen_len steps.  Returns the
        batch slot, or None when no slot or not enough blocks are free."""
        P = int(prompt_k.shape[0])
        rc = lib().decode_engine_admit(self._eng, P, int(gen_len), ctypes.c_void_p(prompt_k.data_ptr()),
                                       ctypes.c_void_p(prompt_v.data_ptr()), ctypes.c_void_p(self.k_cache.data_ptr()),
                                       ctypes.c_void_p(self.v_cache.data_ptr()), ctypes.byref(self._dims),
                                       api._stream(None), ctypes.byref(self._slot))
        if rc == -5:
            return None
        api._check(rc, "decode_engine_admit")
        self._num_free -= 1
        return int(self._slot.value)

    def fork(self, src_slot: int, gen_len: int) -> Optional[int]:
        """Parallel sampling: a new sequence sharing every block of the one in
        src_slot, running gen_len steps.  Returns its batch slot, or None when
        no slot is free."""
        rc = lib().decode_engine_fork(self._eng, int(src_slot), int(gen_len), ctypes.byref(self._slot))
        if rc == -5:
            return None
        api._check(rc, "decode_engine_fork")
        self._num_free -= 1
        return int(self._slot.value)

    # ------------------------------------------------------------------ one step

    def step(self, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor) -> torch.Tensor:
        """One decode step for every active slot (rows of q / k_new / v_new of
        empty slots are ignored).  Returns the [max_batch][Hq][D] output tensor
        (rewritten by the next step)."""
        key = (q.data_ptr(), k_new.data_ptr(), v_new.data_ptr())
        if self._step_args is None or self._step_key != key:
            for n, t in (("q", q), ("k_new", k_new), ("v_new", v_new)):
                api._need_cuda(n, t, self.dtype)
            if q.shape != (self.B, self.H, self.D) or k_new.shape != (self.B, self.Hk, self.D) or \
                    v_new.shape != k_new.shape:
                raise ValueError("q / k_new / v_new must cover every batch slot")
            P = ctypes.c_void_p
            ws = self.workspace
            self._step_args = (self._eng, P(q.data_ptr()), P(k_new.data_ptr()), P(v_new.data_ptr()),
                               P(self.k_cache.data_ptr()), P(self.v_cache.data_ptr()),
                               ctypes.c_float(1.0 / math.sqrt(self.D)), P(self.out.data_ptr()),
                               P(ws.data_ptr() if ws is not None else 0), ws.numel() if ws is not None else 0,
                               ctypes.byref(self._dims))
            self._step_key = key
        api._check(lib().decode_engine_step(*self._step_args, api._stream(None)), "decode_engine_step")
        self.steps += 1
        return self.out

    def finish_step(self) -> list:
        """Count the step against each active sequence; those that finished
        free their blocks.  Returns their former slots."""
        api._check(lib().decode_engine_finish(self._eng, self._freed.ctypes.data_as(c_int32_p),
                                              ctypes.byref(self._nfreed)), "decode_engine_finish")
        n = self._nfreed.value
        self._num_free += n
        return self._freed[:n].tolist()

    # ------------------------------------------------------------------ accounting

    def last_step(self):
        """(block tables int32[max_batch][max_blocks], context lengths
        int32[max_batch]) that the last step ran with."""
        tables = np.empty((self.B, self.max_blocks), np.int32)
        lens = np.empty(self.B, np.int32)
        api._check(lib().decode_engine_last_step(self._eng, tables.ctypes.data_as(c_int32_p),
                                                 lens.ctypes.data_as(c_int32_p)), "decode_engine_last_step")
        return tables, lens

    def stats(self) -> dict:
        """Totals since creation or reset_stats(): steps, tokens generated
        (sequence_steps), tokens attended (context_tokens), unused tail slots
        of the last blocks, copy-on-write block copies."""
        st = PkvEngineStats()
        api._check(lib().decode_engine_get_stats(self._eng, ctypes.byref(st)), "decode_engine_get_stats")
        return {name: int(getattr(st, name)) for name, _ in PkvEngineStats._fields_}

    def reset_stats(self) -> None:
        api._check(lib().decode_engine_reset_stats(self._eng), "decode_engine_reset_stats")

    def context_lengths(self) -> np.ndarray:
        """Current context length of every batch slot (0 = empty)."""
        self._state()
        return self._lens.astype(np.int64)

    def waste_blocks(self) -> float:
        """Mean unused tail of the last block per active sequence, in blocks (< 1)."""
        L = self.context_lengths()
        L = L[L > 0]
        if L.size == 0:
            return 0.0
        return float(((-(-L // BLOCK_SIZE)) * BLOCK_SIZE - L).mean() / BLOCK_SIZE)

"""Shared pieces of the GPU parity tests: run one decode step through the C ABI
and the same step through the fp64 oracle, then compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_cache_26_gb300 as pkv

ATOL, RTOL = 2e-3, 1e-2   # |gpu - ref| <= ATOL + RTOL * |ref|, elementwise


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def run_gpu_step(w, layer=0, num_splits=0, device="cuda", slots=None, fused=False):
    """Append each sequence's new token, then attend: with paged_kv_append +
    paged_decode_attention, or with the single paged_decode_step call when
    ``fused``.  Returns (out, k_cache, v_cache) as CPU tensors; the workload's
    own tensors are not modified."""
    kc = w.k_cache[layer].to(device, copy=True)
    vc = w.v_cache[layer].to(device, copy=True)
    q = w.q[layer].to(device)
    kn = w.k_new[layer].to(device)
    vn = w.v_new[layer].to(device)
    if slots is None:
        slots = pkv.paged_kv_slot_mapping(w.block_tables, w.context_lens, w.spec.block_size)
    slot_t = torch.from_numpy(np.asarray(slots, np.int32)).to(device)
    bt = torch.from_numpy(w.block_tables).to(device)
    cl = torch.from_numpy(w.context_lens).to(device)
    if fused:
        out = pkv.paged_decode_step(q, kn, vn, kc, vc, bt, cl, w.scale, num_splits=num_splits)
    else:
        pkv.paged_kv_append(kn, vn, slot_t, kc, vc)
        out = pkv.paged_decode_attention(q, kc, vc, bt, cl, w.scale, num_splits=num_splits)
    pkv.paged_kv_check_status()
    return out.cpu(), kc.cpu(), vc.cpu()


def oracle_caches(w, layer=0):
    """The caches after the oracle's append of each sequence's newest token."""
    slots = oracle.slot_mapping(w.block_tables, w.context_lens, w.spec.block_size)
    return oracle.kv_append(bits(w.k_cache[layer]), bits(w.v_cache[layer]), bits(w.k_new[layer]),
                            bits(w.v_new[layer]), slots, w.spec.block_size)


def oracle_rows(w, kc_bits, vc_bits, rows, layer=0):
    return oracle.decode_attention_rows(bits(w.q[layer]), kc_bits, vc_bits, w.block_tables, w.context_lens,
                                        w.scale, w.spec.dtype, w.spec.block_size, rows)


def widen_out(out: torch.Tensor, dtype: str) -> np.ndarray:
    return oracle.widen(bits(out), dtype)


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU output"
    err = np.abs(gpu - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {err.size} outside tolerance; worst at {i}: "
                             f"gpu={gpu[i]!r} ref={ref[i]!r} err={err[i]:.3e} bound={bound[i]:.3e}")


def sample_rows(w, n, seed=0):
    """n (sequence, query head) pairs: the longest and shortest sequences, the
    shared-prefix and spiked ones, then seeded random picks."""
    B, H = w.spec.batch, w.spec.num_q_heads
    rng = np.random.default_rng(seed)
    picks = {(int(np.argmax(w.context_lens)), 0), (int(np.argmin(w.context_lens)), H - 1)}
    for b in list(w.shared_seqs[:2]):
        picks.add((int(b), int(rng.integers(H))))
    while len(picks) < min(n, B * H):
        picks.add((int(rng.integers(B)), int(rng.integers(H))))
    return sorted(picks)


def oracle_all_rows(w, kc_bits, vc_bits, layer=0):
    """Every (sequence, query head) output of the oracle, float64 [B][Hq][D].
    The same definition as oracle.decode_attention_rows (gather through the
    table, then softmax(scale q K^T) V in fp64), but each (sequence, KV head)
    is gathered once and shared by its group's query heads, which keeps
    full-size configurations to seconds."""
    s = w.spec
    B, H, D, g = s.batch, s.num_q_heads, s.head_dim, s.group
    q = oracle.widen(bits(w.q[layer]), s.dtype)
    out = np.zeros((B, H, D))
    for b in range(B):
        L = int(w.context_lens[b])
        if L == 0:
            continue
        for kvh in range(s.num_kv_heads):
            K = oracle.widen(oracle.gather_kv(kc_bits, w.block_tables[b], L, kvh, s.block_size), s.dtype)
            V = oracle.widen(oracle.gather_kv(vc_bits, w.block_tables[b], L, kvh, s.block_size), s.dtype)
            for h in range(kvh * g, (kvh + 1) * g):
                out[b, h] = oracle.attend_one(q[b, h], K, V, w.scale)[0]
    return out

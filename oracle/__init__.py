"""fp64 CPU oracle for paged decode attention and the per-step KV append.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this package; only
the tests, the smoke check in ``__graft_entry__`` and the CPU-baseline leg of
``bench.py`` may use it.  It shares no code with the CUDA path (no kernels,
headers, helpers or tables): both sides are fed the same seeded inputs and the
tests compare what each produces.

Everything here is written from the pages' statement of the method, in numpy,
in float64, one (sequence, query head) at a time, so that a reader can check it
against the pages by eye:

* Decode attention is the plain definition softmax(q K^T * scale) V for the one
  new query token, with no mask (youngju.dev "LLM サービング最適化完全ガイド",
  the ``AttentionWithKVCache`` listing: scores = Q K^T / sqrt(d_k), softmax,
  weights V).  The API's ``scale`` multiplies the scores; passing
  1/sqrt(head_dim) gives the listing's division by sqrt(d_k).
* K and V are read through the block table: logical block j of a sequence lives
  in physical block table[j] (kasblo.com "vLLMとは？", section
  "PagedAttentionはKV Cacheをblockで管理する": A0->7, A1->1, A2->9 and "the
  attention kernel reads the K/V it needs by consulting this table").
* Grouped-query attention: query heads [kv*g, (kv+1)*g) share KV head kv
  (notes on "How to Scale Your Model, Part 7: Inference", section
  "生成スループット/レイテンシ改善のテクニック", GQA figure; design.babushkai.com
  "GPU推論の内部構造", section "KVキャッシュの台帳").
* The append stores the new token's K/V at its slot so later steps reuse it
  ("How to Scale Your Model, Part 7", section "Transformer 推論の基礎: Prefill と
  Generation": the new token's KV projection is appended to the cache).
* The split / log-sum-exp merge follows from the online softmax of FlashAttention
  (design.babushkai.com "GPU推論の内部構造", section "カーネル: FlashAttentionと
  メモリ階層"): each split is a normalised partial result plus its log-sum-exp.
* KV-size accounting follows the worked formulas of kasblo.com "vLLMとは？",
  section "KV Cacheの容量をtokenから計算する", and the roofline step-time model of
  design.babushkai.com "GPU推論の内部構造", section "バッチングの経済学".

Inputs that carry fp16/bf16 values arrive as their raw 16-bit patterns
(``np.uint16``) and are widened here to float64, so the oracle sees exactly the
rounded values the GPU sees.
"""
from __future__ import annotations

import math
from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np

__all__ = [
    "widen", "e4m3_decode", "e4m3_encode", "quantize_e4m3", "dequantize_e4m3", "kv_append_fp8", "kv_head_of", "slot_of_position", "slot_mapping", "kv_append",
    "gather_kv", "attend_one", "decode_attention", "decode_attention_rows", "decode_attention_multi",
    "slot_mapping_multi", "copy_blocks",
    "split_partials", "lse_merge", "kv_bytes_per_token", "blocks_needed",
    "allocated_bytes", "wasted_bytes", "kv_cache_bytes", "decode_step_tokens_per_s",
    "attention_call_bytes",
]


# ---------------------------------------------------------------- number formats

def widen(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of each fp16 / bf16 bit pattern.

    fp16 is IEEE-754 binary16 (numpy implements it).  bf16 is by definition the
    upper 16 bits of an IEEE-754 binary32, so the pattern shifted left by 16 and
    read as float32 is its value.
    """
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "fp16":
        return bits.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


# ---------------------------------------------------------------- fp8 (E4M3) KV codes
#
# The FP8 KV cache (design.babushkai.com "GPU推論の内部構造", section "KVキャッシュの
# 台帳", and youngju.dev, quantization section: an FP8 KV cache halves the
# bytes per token) stores each K/V element as an E4M3 code with one float32
# scale per KV head: value = decode(code) * scale.  E4M3 as used for FP8 KV
# caches: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no
# infinities, S.1111.111 = NaN, largest finite 448, subnormals k * 2^-9.

E4M3_MAX = 448.0


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Exact float64 value of each E4M3 code (NaN for S.1111.111)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e4m3_encode(x) -> np.ndarray:
    """E4M3 code of each float32 value: round to nearest, ties to even;
    magnitudes beyond 448 saturate to 448; NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)   # exact
    out = np.zeros(x.shape, dtype=np.uint8)
    sign = (np.signbit(x)).astype(np.uint8) << 7
    a = np.abs(x)
    nan = np.isnan(x)
    # grid spacing at |x|: 2^-9 below the smallest normal 2^-6, else 2^(e-3)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.clip(e, -6, 8)
    step = 2.0 ** (e - 3)
    q = np.rint(a / step) * step          # nearest multiple, ties to even (exact in float64)
    q = np.minimum(q, E4M3_MAX)           # saturate (also catches rounding up past 448)
    # code of the (representable) magnitude q
    qe = np.floor(np.log2(np.where(q > 0, q, 1.0)))
    normal = q >= 2.0 ** -6
    exp_field = np.where(normal, qe + 7, 0)
    mant = np.where(normal, np.rint((q / 2.0 ** qe - 1.0) * 8), np.rint(q / 2.0 ** -9))
    code = (exp_field.astype(np.int64) << 3) | mant.astype(np.int64)
    out[:] = np.where(nan, 0x7F, code | sign.astype(np.int64))
    return out


def quantize_e4m3(bits: np.ndarray, dtype: str, scale: float) -> np.ndarray:
    """The append's quantisation of fp16/bf16 values with a float32 scale:
    code = e4m3(float32(x) / float32(scale)), the division in float32."""
    x = widen(bits, dtype).astype(np.float32)                 # exact: fp16/bf16 fit in float32
    y = x / np.float32(scale)                                 # IEEE float32 division
    return e4m3_encode(y)


def dequantize_e4m3(codes: np.ndarray, scale: float) -> np.ndarray:
    return e4m3_decode(codes) * float(np.float32(scale))


# ---------------------------------------------------------------- indexing

def kv_head_of(q_head: int, group: int) -> int:
    """Query head h reads KV head h // g (contiguous grouping)."""
    return q_head // group


def slot_of_position(table_row: np.ndarray, pos: int, block_size: int) -> int:
    """Physical slot of token position ``pos``: block table[pos // BS], offset pos % BS."""
    return int(table_row[pos // block_size]) * block_size + pos % block_size


def slot_mapping(block_tables: np.ndarray, context_lens: np.ndarray, block_size: int) -> np.ndarray:
    """Slot of each sequence's newest token (position L-1); -1 when L == 0."""
    out = np.full(len(context_lens), -1, dtype=np.int32)
    for b, L in enumerate(np.asarray(context_lens)):
        if L > 0:
            out[b] = slot_of_position(block_tables[b], int(L) - 1, block_size)
    return out


# ---------------------------------------------------------------- append

def kv_append_fp8(k_cache: np.ndarray, v_cache: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
                  slots: np.ndarray, block_size: int, k_scale: np.ndarray, v_scale: np.ndarray,
                  dtype: str) -> Tuple[np.ndarray, np.ndarray]:
    """kv_append into E4M3 caches: token i's K/V of KV head h are quantised with
    k_scale[h] / v_scale[h] before they are stored."""
    Hkv = k_new.shape[1]
    kq = np.stack([quantize_e4m3(k_new[:, h], dtype, k_scale[h]) for h in range(Hkv)], axis=1)
    vq = np.stack([quantize_e4m3(v_new[:, h], dtype, v_scale[h]) for h in range(Hkv)], axis=1)
    return kv_append(k_cache, v_cache, kq, vq, slots, block_size)


def kv_append(k_cache: np.ndarray, v_cache: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
              slots: np.ndarray, block_size: int) -> Tuple[np.ndarray, np.ndarray]:
    """Copies of the caches with token i's K/V (all KV heads) stored at slot[i].

    Caches are [num_blocks][num_kv_heads][block_size][head_dim] bit patterns;
    k_new / v_new are [num_tokens][num_kv_heads][head_dim].  A negative slot
    means "no token to store".
    """
    k_out = np.array(k_cache, copy=True)
    v_out = np.array(v_cache, copy=True)
    for i, slot in enumerate(np.asarray(slots)):
        if slot < 0:
            continue
        blk, off = divmod(int(slot), block_size)
        k_out[blk, :, off, :] = k_new[i]
        v_out[blk, :, off, :] = v_new[i]
    return k_out, v_out


# ---------------------------------------------------------------- attention

def gather_kv(cache: np.ndarray, table_row: np.ndarray, ctx: int, kv_head: int, block_size: int) -> np.ndarray:
    """Contiguous [ctx][head_dim] copy of one sequence's K (or V) for one KV head,
    token t read from physical block table_row[t // BS] at offset t % BS."""
    t = np.arange(ctx)
    blocks = np.asarray(table_row, dtype=np.int64)[t // block_size]
    return cache[blocks, kv_head, t % block_size, :]


def attend_one(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """softmax(scale * K q) V for one query vector, in float64.

    Returns (output[D], weights[L], log-sum-exp of the scaled scores).
    """
    s = scale * (K * q[None, :]).sum(axis=1)
    m = s.max()
    e = np.exp(s - m)
    z = e.sum()
    p = e / z
    o = (p[:, None] * V).sum(axis=0)
    return o, p, m + math.log(z)


def _dims(q_bits, k_cache_bits):
    B, Hq, D = q_bits.shape
    Hkv = k_cache_bits.shape[1]
    if Hq % Hkv:
        raise ValueError("num_kv_heads must divide num_q_heads")
    return B, Hq, Hkv, D


def decode_attention_rows(q_bits, k_cache_bits, v_cache_bits, block_tables, context_lens,
                          scale: float, dtype: str, block_size: int,
                          rows: Iterable[Tuple[int, int]], kv_scales=None) -> np.ndarray:
    """Attention output (float64 [len(rows)][D]) for the listed (sequence, query head) pairs.

    With ``kv_scales = (k_scale, v_scale)`` the caches hold E4M3 codes and the
    attention runs on their dequantised values (code value * the KV head's scale)."""
    B, Hq, Hkv, D = _dims(q_bits, k_cache_bits)
    g = Hq // Hkv
    rows = list(rows)
    out = np.zeros((len(rows), D), dtype=np.float64)
    for i, (b, h) in enumerate(rows):
        L = int(context_lens[b])
        if L == 0:
            continue  # empty context: output stays zero
        kv = kv_head_of(h, g)
        if kv_scales is None:
            K = widen(gather_kv(k_cache_bits, block_tables[b], L, kv, block_size), dtype)
            V = widen(gather_kv(v_cache_bits, block_tables[b], L, kv, block_size), dtype)
        else:
            K = dequantize_e4m3(gather_kv(k_cache_bits, block_tables[b], L, kv, block_size), kv_scales[0][kv])
            V = dequantize_e4m3(gather_kv(v_cache_bits, block_tables[b], L, kv, block_size), kv_scales[1][kv])
        q = widen(q_bits[b, h], dtype)
        out[i] = attend_one(q, K, V, scale)[0]
    return out


def decode_attention(q_bits, k_cache_bits, v_cache_bits, block_tables, context_lens,
                     scale: float, dtype: str, block_size: int) -> np.ndarray:
    """Attention output float64 [B][Hq][D] for every sequence and query head."""
    B, Hq, Hkv, D = _dims(q_bits, k_cache_bits)
    rows = [(b, h) for b in range(B) for h in range(Hq)]
    return decode_attention_rows(q_bits, k_cache_bits, v_cache_bits, block_tables, context_lens,
                                 scale, dtype, block_size, rows).reshape(B, Hq, D)


# ---------------------------------------------------------------- copy-on-write

def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray, pairs) -> Tuple[np.ndarray, np.ndarray]:
    """Copy-on-write of shared blocks (kasblo.com "vLLMとは？", section
    "block共有とAutomatic Prefix Caching": a block shared by several sequences is
    duplicated only when one of them must write into it).  For each (src, dst)
    pair, physical block dst becomes a copy of block src (every KV head, every
    slot, K and V).  Destinations are distinct and are not sources."""
    k = k_cache.copy()
    v = v_cache.copy()
    for src, dst in pairs:
        k[dst] = k_cache[src]
        v[dst] = v_cache[src]
    return k, v


# ---------------------------------------------------------------- several new tokens per sequence

def decode_attention_multi(q_bits, k_cache_bits, v_cache_bits, block_tables, context_lens, q_len: int,
                           scale: float, dtype: str, block_size: int, kv_scales=None,
                           rows: Optional[Iterable[Tuple[int, int, int]]] = None) -> np.ndarray:
    """Decode attention for q_len new tokens per sequence (speculative
    verification, chunked decode: youngju.dev "LLM サービング最適化完全ガイド",
    speculative decoding section -- the target model checks several draft
    tokens in one pass -- and design.babushkai.com "GPU推論の内部構造", section
    "KVキャッシュの台帳", chunked prefill).

    q_bits: [B][q_len][Hq][D].  context_lens[b] = L counts the q_len new tokens,
    which sit at positions L - q_len .. L - 1; new token i attends to positions
    [0, L - q_len + i] (causal among the new tokens).  A token whose position
    is negative (L < q_len) attends to nothing and gets a zero row.

    Returns float64 [B][q_len][Hq][D], or, for ``rows`` = [(b, i, h), ...],
    float64 [len(rows)][D]."""
    q_bits = np.asarray(q_bits)
    B, n, Hq, D = q_bits.shape
    Hkv = k_cache_bits.shape[1]
    g = Hq // Hkv
    want = rows if rows is not None else [(b, i, h) for b in range(B) for i in range(n) for h in range(Hq)]
    out = np.zeros((len(want), D))
    for r, (b, i, h) in enumerate(want):
        pos = int(context_lens[b]) - n + i
        if pos < 0:
            continue
        kv = kv_head_of(h, g)
        Kc = gather_kv(k_cache_bits, block_tables[b], pos + 1, kv, block_size)
        Vc = gather_kv(v_cache_bits, block_tables[b], pos + 1, kv, block_size)
        if kv_scales is None:
            K, V = widen(Kc, dtype), widen(Vc, dtype)
        else:
            K, V = dequantize_e4m3(Kc, kv_scales[0][kv]), dequantize_e4m3(Vc, kv_scales[1][kv])
        out[r] = attend_one(widen(q_bits[b, i, h], dtype), K, V, scale)[0]
    return out if rows is not None else out.reshape(B, n, Hq, D)


def slot_mapping_multi(block_tables, context_lens, q_len: int, block_size: int) -> np.ndarray:
    """Slots of each sequence's q_len newest tokens (positions L - q_len .. L - 1),
    int32 [B][q_len]; -1 for a position below 0."""
    B = len(context_lens)
    out = np.full((B, q_len), -1, dtype=np.int32)
    for b in range(B):
        for i in range(q_len):
            pos = int(context_lens[b]) - q_len + i
            if pos >= 0:
                out[b, i] = slot_of_position(block_tables[b], pos, block_size)
    return out


# ---------------------------------------------------------------- split + merge

def split_partials(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float,
                   split_tokens: int) -> List[Tuple[np.ndarray, float]]:
    """Per split of ``split_tokens`` consecutive keys: (normalised output, log-sum-exp).

    A split holding no key contributes (zeros, -inf).
    """
    L = K.shape[0]
    n = max(1, -(-L // split_tokens))
    parts = []
    for s in range(n):
        lo, hi = s * split_tokens, min(L, (s + 1) * split_tokens)
        if hi <= lo:
            parts.append((np.zeros(K.shape[1]), -math.inf))
            continue
        o, _, lse = attend_one(q, K[lo:hi], V[lo:hi], scale)
        parts.append((o, lse))
    return parts


def lse_merge(parts: Sequence[Tuple[np.ndarray, float]]) -> np.ndarray:
    """Combine normalised partial outputs by their log-sum-exp weights:
    out = sum_s exp(lse_s - M) o_s / sum_s exp(lse_s - M), M = max_s lse_s."""
    lses = np.array([p[1] for p in parts], dtype=np.float64)
    M = lses.max()
    if M == -math.inf:
        return np.zeros_like(parts[0][0])
    w = np.exp(lses - M)
    return sum(wi * o for wi, (o, _) in zip(w, parts)) / w.sum()


# ---------------------------------------------------------------- accounting

def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    """m_token = 2 L H_kv d_h b (K and V)."""
    return 2 * layers * kv_heads * head_dim * elem_bytes


def blocks_needed(tokens: int, block_size: int) -> int:
    """n_blocks = ceil(N / B)."""
    return -(-tokens // block_size)


def allocated_bytes(tokens: int, block_size: int, m_token: int) -> int:
    """M_alloc = ceil(N / B) * B * m_token."""
    return blocks_needed(tokens, block_size) * block_size * m_token


def wasted_bytes(tokens: int, block_size: int, m_token: int) -> int:
    """M_waste = (ceil(N / B) * B - N) * m_token: the unused tail of the last block."""
    return (blocks_needed(tokens, block_size) * block_size - tokens) * m_token


def kv_cache_bytes(seq_len: int, n_layers: int, n_kv_heads: int, head_dim: int,
                   batch_size: int, dtype_bytes: int = 2) -> int:
    """2 (K and V) x layers x KV heads x head_dim x tokens x batch x bytes."""
    return 2 * n_layers * n_kv_heads * head_dim * seq_len * batch_size * dtype_bytes


def decode_step_tokens_per_s(batch: int, ctx: int, bandwidth: float, compute: float,
                             weight_bytes: float, kv_bytes_per_tok: float, params: float) -> float:
    """Roofline decode step: time = max(bytes / BW, flops / peak), where the
    weights are read once per step and every sequence reads its own KV;
    returns batch / time (tokens per second for the whole batch)."""
    bytes_moved = weight_bytes + batch * ctx * kv_bytes_per_tok
    flops = batch * 2 * params
    return batch / max(bytes_moved / bandwidth, flops / compute)


def attention_call_bytes(context_lens, batch: int, num_q_heads: int, num_kv_heads: int,
                         head_dim: int, elem_bytes: int, table_entries_read: int) -> int:
    """Algorithmic HBM bytes of one decode-attention call: the K and V of every
    cached token for every KV head, plus q, out, the block-table entries read
    and the context lengths (int32)."""
    kv = int(np.asarray(context_lens, np.int64).sum()) * num_kv_heads * head_dim * 2 * elem_bytes
    q_out = 2 * batch * num_q_heads * head_dim * elem_bytes
    return kv + q_out + 4 * table_entries_read + 4 * batch

"""Seeded synthetic inputs for paged decode attention and the per-step KV append.

This module only draws inputs: sequence lengths, the scattered placement of
physical blocks, block tables, and N(0,1) values for q, the KV pool and the new
token's K/V.  It holds none of the attention arithmetic, so both the CUDA path
and the fp64 oracle can be fed from it without sharing any of the method.

Shapes follow the vLLM-style paged layout (pages: kasblo.com "What is vLLM /
PagedAttention", section "PagedAttention manages the KV cache in blocks";
youngju.dev "LLM serving optimization complete guide", PagedAttention memory
layout figure):

  k_cache, v_cache : T[num_blocks][num_kv_heads][block_size][head_dim]
  q                : T[batch][num_q_heads][head_dim]
  k_new, v_new     : T[batch][num_kv_heads][head_dim]   (one new token per sequence)
  block_tables     : int32[batch][max_blocks]           (-1 past a sequence's last block)
  context_lens     : int32[batch]                       (includes the new token)

Every cache slot that does not hold one of the first ``context_len - 1`` tokens
of some sequence (free blocks, the tail of each last block, and the slot the
append will fill) is set to NaN.  A kernel that reads past a sequence's length
therefore shows up as NaN in its output instead of passing by luck.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class WorkloadSpec:
    """Shape and distribution of one synthetic decode batch."""

    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: str  # "fp16" | "bf16"
    # ("fixed", (l0, l1, ...)) | ("constant", L) | ("uniform", lo, hi)
    # | ("lognormal", median, sigma, lo, hi)
    lengths: tuple
    block_size: int = 16
    # ("fixed", num_blocks) | ("factor", f): pool = ceil(f * unique blocks needed)
    pool: tuple = ("factor", 1.25)
    num_layers: int = 1
    # (num_sharing_seqs, prefix_tokens): that many sequences point their first
    # prefix_tokens/block_size table entries at the same physical blocks.
    shared_prefix: Optional[Tuple[int, int]] = None
    # logit value planted at one seeded key position per sequence (None = off)
    spike_logit: Optional[float] = None
    # split size (tokens) the configuration is quoted with; None = single pass
    split_tokens: Optional[int] = None

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def replace(self, **kw) -> "WorkloadSpec":
        return dataclasses.replace(self, **kw)


# The five configurations the measurements are quoted on.
TINY = WorkloadSpec(
    name="tiny", batch=4, num_q_heads=8, num_kv_heads=2, head_dim=64, dtype="fp16",
    lengths=("fixed", (17, 40, 64, 100)), pool=("fixed", 32))
LLAMA3_8B = WorkloadSpec(
    name="llama3_8b_b64", batch=64, num_q_heads=32, num_kv_heads=8, head_dim=128,
    dtype="bf16", lengths=("uniform", 512, 4096))
MHA_7B_B16 = WorkloadSpec(
    name="mha7b_b16_s2048", batch=16, num_q_heads=32, num_kv_heads=32, head_dim=128,
    dtype="fp16", lengths=("constant", 2048), num_layers=32)
MHA_7B_B64 = WorkloadSpec(
    name="mha7b_b64_s4096", batch=64, num_q_heads=32, num_kv_heads=32, head_dim=128,
    dtype="fp16", lengths=("constant", 4096), num_layers=32)
LLAMA70B_TAIL = WorkloadSpec(
    name="llama70b_tail_b256", batch=256, num_q_heads=64, num_kv_heads=8, head_dim=128,
    dtype="bf16", lengths=("lognormal", 1000.0, 1.0, 80, 8192),
    shared_prefix=(64, 512))
LONG_CTX = WorkloadSpec(
    name="longctx_b8_32k", batch=8, num_q_heads=32, num_kv_heads=8, head_dim=128,
    dtype="bf16", lengths=("constant", 32768), spike_logit=8.0, split_tokens=512)

CONFIGS = {s.name: s for s in (TINY, LLAMA3_8B, MHA_7B_B16, MHA_7B_B64, LLAMA70B_TAIL, LONG_CTX)}


@dataclass
class Workload:
    spec: WorkloadSpec
    seed: int
    context_lens: np.ndarray          # int32[B], includes the appended token
    block_tables: np.ndarray          # int32[B][MB], -1 padded
    num_blocks: int
    scale: float
    q: List[torch.Tensor]             # per layer: T[B][Hq][D]
    k_new: List[torch.Tensor]         # per layer: T[B][Hkv][D]
    v_new: List[torch.Tensor]
    k_cache: List[torch.Tensor]       # per layer: T[NB][Hkv][BS][D], before the append
    v_cache: List[torch.Tensor]
    shared_seqs: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int64))
    spike_pos: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int64))

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])


def draw_lengths(spec: WorkloadSpec, rng: np.random.Generator) -> np.ndarray:
    kind = spec.lengths[0]
    if kind == "fixed":
        lens = np.asarray(spec.lengths[1], dtype=np.int64)
        assert lens.shape == (spec.batch,)
    elif kind == "constant":
        lens = np.full(spec.batch, int(spec.lengths[1]), dtype=np.int64)
    elif kind == "uniform":
        lo, hi = spec.lengths[1], spec.lengths[2]
        lens = rng.integers(lo, hi + 1, size=spec.batch, dtype=np.int64)
    elif kind == "lognormal":
        median, sigma, lo, hi = spec.lengths[1:]
        raw = rng.lognormal(mean=math.log(median), sigma=sigma, size=spec.batch)
        lens = np.clip(np.rint(raw), lo, hi).astype(np.int64)
    else:
        raise ValueError(f"unknown length distribution {kind!r}")
    return lens


def _cdiv(a, b):
    return -(-a // b)


def generate(spec: WorkloadSpec, seed: int = 0, device="cpu", layers: Optional[int] = None,
             new_tokens: int = 1) -> Workload:
    """Draw one decode batch.  ``layers`` caps the number of layer caches built
    (the structure, i.e. lengths and tables, is the same for every layer).
    ``new_tokens``: tokens each sequence appends this step; a sequence sharing
    the prefix holds at least prefix + new_tokens tokens, so that its new
    tokens never land in a shared block."""
    rng = np.random.default_rng(seed)
    bs = spec.block_size
    lens = draw_lengths(spec, rng)

    shared_seqs = np.zeros(0, np.int64)
    prefix_blocks = 0
    if spec.shared_prefix is not None:
        n_share, prefix_tokens = spec.shared_prefix
        assert prefix_tokens % bs == 0, "shared prefix must cover whole blocks"
        prefix_blocks = prefix_tokens // bs
        eligible = np.flatnonzero(lens >= prefix_tokens + new_tokens)
        if eligible.size >= n_share:
            shared_seqs = np.sort(rng.choice(eligible, size=n_share, replace=False))
        else:
            shared_seqs = np.sort(rng.choice(spec.batch, size=n_share, replace=False))
            lens[shared_seqs] = np.maximum(lens[shared_seqs], prefix_tokens + new_tokens)

    nblk = _cdiv(lens, bs)
    is_shared = np.zeros(spec.batch, bool)
    is_shared[shared_seqs] = True
    private = nblk - np.where(is_shared, prefix_blocks, 0)
    unique_needed = int(private.sum()) + (prefix_blocks if shared_seqs.size else 0)
    if spec.pool[0] == "fixed":
        num_blocks = int(spec.pool[1])
    else:
        num_blocks = max(1, int(math.ceil(spec.pool[1] * unique_needed)))
    assert num_blocks >= unique_needed, "pool too small for the batch"

    # Scattered physical placement: walk a seeded permutation of the pool.
    perm = rng.permutation(num_blocks).astype(np.int64)
    cursor = 0
    shared_ids = perm[cursor:cursor + prefix_blocks] if shared_seqs.size else np.zeros(0, np.int64)
    cursor += shared_ids.size
    mb = int(nblk.max())
    tables = np.full((spec.batch, mb), -1, dtype=np.int32)
    for b in range(spec.batch):
        first = 0
        if is_shared[b]:
            tables[b, :prefix_blocks] = shared_ids
            first = prefix_blocks
        n = int(nblk[b]) - first
        tables[b, first:first + n] = perm[cursor:cursor + n]
        cursor += n

    dt = DTYPES[spec.dtype]
    nl = spec.num_layers if layers is None else min(layers, spec.num_layers)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    scale = 1.0 / math.sqrt(spec.head_dim)

    # Slots holding one of the first L-1 tokens of some sequence.
    tok_blocks, tok_offs = [], []
    for b in range(spec.batch):
        t = np.arange(int(lens[b]) - 1, dtype=np.int64)
        tok_blocks.append(tables[b, t // bs].astype(np.int64))
        tok_offs.append(t % bs)
    valid = np.zeros((num_blocks, bs), bool)
    valid[np.concatenate(tok_blocks), np.concatenate(tok_offs)] = True
    invalid = torch.from_numpy(~valid).to(device)

    spike_pos = np.zeros(0, np.int64)
    if spec.spike_logit is not None:
        spike_pos = np.array([rng.integers(0, int(lens[b])) for b in range(spec.batch)], np.int64)

    def randn(shape):
        return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(dt)

    qs, kn, vn, kc, vc = [], [], [], [], []
    H, Hk, D = spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    for _ in range(nl):
        kcache = randn((num_blocks, Hk, bs, D))
        vcache = randn((num_blocks, Hk, bs, D))
        kcache.permute(0, 2, 1, 3)[invalid] = float("nan")
        vcache.permute(0, 2, 1, 3)[invalid] = float("nan")
        q = randn((spec.batch, H, D))
        k_new = randn((spec.batch, Hk, D))
        v_new = randn((spec.batch, Hk, D))
        if spec.spike_logit is not None:
            _plant_spikes(spec, scale, q, k_new, kcache, tables, lens, spike_pos)
        qs.append(q); kn.append(k_new); vn.append(v_new); kc.append(kcache); vc.append(vcache)

    return Workload(spec=spec, seed=seed, context_lens=lens.astype(np.int32), block_tables=tables,
                    num_blocks=num_blocks, scale=scale, q=qs, k_new=kn, v_new=vn,
                    k_cache=kc, v_cache=vc, shared_seqs=shared_seqs, spike_pos=spike_pos)


def _plant_spikes(spec, scale, q, k_new, kcache, tables, lens, spike_pos):
    """Place one key per sequence and KV head whose logit against the first
    query head of the group is ``spike_logit`` (before rounding to T)."""
    g = spec.group
    bs = spec.block_size
    for b in range(spec.batch):
        p = int(spike_pos[b])
        for h in range(spec.num_kv_heads):
            qv = q[b, h * g].to(torch.float64)
            key = (spec.spike_logit * qv / (scale * torch.dot(qv, qv))).to(q.dtype)
            if p == int(lens[b]) - 1:
                k_new[b, h] = key
            else:
                kcache[int(tables[b, p // bs]), h, p % bs] = key



# ---------------------------------------------------------------- E4M3 pools

@dataclass
class Fp8Caches:
    """E4M3 stand-ins of a workload's caches (before the append)."""

    k_cache: List[torch.Tensor]   # per layer: uint8[NB][Hkv][BS][D], E4M3 codes
    v_cache: List[torch.Tensor]
    k_scale: List[torch.Tensor]   # per layer: float32[Hkv]
    v_scale: List[torch.Tensor]


def fp8_caches(w: Workload, seed: int = 0) -> Fp8Caches:
    """Draw an E4M3 pool for workload ``w``: per layer and KV head a K scale and
    a V scale drawn uniformly from [0.004, 0.02], and as codes the workload's own
    N(0,1) cache values over those scales, cast by torch's float8_e4m3fn
    conversion after clamping to +-448 (so values up to ~1.8-9 sigma are
    represented and the rest sit at +-448).  Every non-token slot holds the NaN
    code 0x7F.  The new token's K/V (``w.k_new`` / ``w.v_new``) stay fp16/bf16:
    the append quantises them."""
    rng = np.random.default_rng(seed + 7919)
    Hk = w.spec.num_kv_heads
    out = Fp8Caches([], [], [], [])
    for layer in range(len(w.k_cache)):
        for src, codes, scales in ((w.k_cache[layer], out.k_cache, out.k_scale),
                                   (w.v_cache[layer], out.v_cache, out.v_scale)):
            s = torch.from_numpy(rng.uniform(0.004, 0.02, Hk).astype(np.float32)).to(src.device)
            x = src.float() / s.view(1, Hk, 1, 1)
            c = x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
            c[torch.isnan(x)] = 0x7F
            codes.append(c)
            scales.append(s)
    return out


# ---------------------------------------------------------------- several new tokens per sequence

@dataclass
class MultiTokens:
    """q_len new tokens per sequence: their queries and K/V rows."""

    q_len: int
    q: List[torch.Tensor]        # per layer: T[B][q_len][Hq][D]
    k_new: List[torch.Tensor]    # per layer: T[B][q_len][Hkv][D]
    v_new: List[torch.Tensor]


def generate_multi(spec: WorkloadSpec, q_len: int, seed: int = 0, device="cpu",
                   layers: Optional[int] = None) -> Tuple[Workload, MultiTokens]:
    """A workload whose sequences each receive q_len new tokens this step: the
    cache holds the first L - q_len tokens of each sequence and NaN in every
    other slot (the q_len slots the append fills included); the new tokens'
    queries and K/V are N(0,1) like the rest."""
    w = generate(spec, seed=seed, device=device, layers=layers, new_tokens=q_len)
    bs = spec.block_size
    blk, off = [], []
    for b in range(spec.batch):
        L = int(w.context_lens[b])
        for pos in range(max(0, L - q_len), L - 1):      # position L - 1 is already NaN
            blk.append(int(w.block_tables[b, pos // bs]))
            off.append(pos % bs)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 104729)
    dt = DTYPES[spec.dtype]
    B, H, Hk, D = spec.batch, spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    m = MultiTokens(q_len, [], [], [])
    for layer in range(len(w.k_cache)):
        if blk:
            bi = torch.tensor(blk, device=device)
            oi = torch.tensor(off, device=device)
            w.k_cache[layer][bi, :, oi, :] = float("nan")
            w.v_cache[layer][bi, :, oi, :] = float("nan")
        m.q.append(torch.randn((B, q_len, H, D), generator=gen, device=device, dtype=torch.float32).to(dt))
        m.k_new.append(torch.randn((B, q_len, Hk, D), generator=gen, device=device, dtype=torch.float32).to(dt))
        m.v_new.append(torch.randn((B, q_len, Hk, D), generator=gen, device=device, dtype=torch.float32).to(dt))
    return w, m

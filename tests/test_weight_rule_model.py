"""Host model of how the multi-token row kernel rounds its softmax weights
(WarpAttnRows in multi_query.cuh, restated in numpy), checked against the
attention tolerance |out - ref| <= 2e-3 + 1e-2 |ref|.

With bf16 inputs the P V product takes each weight p as hi = bf16(p), plus the
remainder lo = bf16(p - hi) only in softmax steps whose weights hold more
than kLoShare of the running sum (any of a warp's 16 rows deciding for the
warp); the normaliser sums the unrounded weights, and a row's reference
maximum moves only when a step's maximum passes it by more than kLazy (log2
units).  Steps are 32 tokens when a KV head has more than 48 query rows, else
16.  The two constants are read from the kernel source, so the model follows
the kernel.  This is a model of the rounding, not of the kernel's exact bits
(scores are taken in fp32 from an fp64 product, the kernel accumulates them
in fp32 on the tensor cores); the GPU parity tests check the kernel itself.
"""
import os
import re

import numpy as np
import torch

import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
with open(os.path.join(ROOT, "paged_kv_cache_26_gb300", "csrc", "multi_query.cuh")) as _f:
    _SRC = _f.read()
LO_SHARE = float(re.search(r"kLoShare\s*=\s*([0-9.]+)f", _SRC).group(1))
LAZY = float(re.search(r"kLazy\s*=\s*([0-9.]+)f", _SRC).group(1))


def _bf16(x):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def _unit_output(rows, K, V, scale, last, share):
    """Model output of one (sequence, KV head): rows [R][D] token-major, the
    unit's K, V [L][D], last[r] = the last position row r attends to; share
    None: no remainder at all."""
    R, L = rows.shape[0], K.shape[0]
    step = 32 if R > 48 else 16
    c2 = scale / np.log(2.0)
    s = (rows @ K.T).astype(np.float32).astype(np.float64)
    s = np.where(np.arange(L)[None, :] <= last[:, None], s, -np.inf)
    m = np.full(R, -np.inf)
    l = np.zeros(R)
    o = np.zeros((R, V.shape[1]))
    warps = (R + 15) // 16
    for t0 in range(0, L, step):
        x = s[:, t0:t0 + step]
        mx = x.max(1) * c2
        up = mx > m + LAZY
        alpha = np.ones(R)
        moved = up & np.isfinite(m)
        alpha[moved] = np.exp2(m[moved] - mx[moved])
        l *= alpha
        o *= alpha[:, None]
        m = np.where(up, mx, m)
        ref = np.where(np.isinf(m), 0.0, m)
        with np.errstate(invalid="ignore"):
            p = np.exp2(x * c2 - ref[:, None])
        p = np.where(np.isfinite(p), p, 0.0).astype(np.float32).astype(np.float64)
        hi = _bf16(p)
        step_sum = p.sum(1)
        row_needs = np.zeros(R, bool) if share is None else step_sum > share * (l + step_sum)
        warp_needs = np.array([row_needs[16 * w:16 * w + 16].any() for w in range(warps)])
        needs = np.repeat(warp_needs, 16)[:R]
        lo = np.where(needs[:, None], _bf16(p - hi), 0.0)
        o += (hi + lo) @ V[t0:t0 + step]
        l += step_sum
    return _bf16(o / np.where(l > 0, l, 1.0)[:, None])


def _worst_over_bound(spec, q_len, seed, share):
    w, m = wl.generate_multi(spec, q_len, seed=seed)
    s = w.spec
    g = s.num_q_heads // s.num_kv_heads
    q = m.q[0].double().numpy()
    kn, vn = m.k_new[0].double().numpy(), m.v_new[0].double().numpy()
    kc, vc = w.k_cache[0].double().numpy(), w.v_cache[0].double().numpy()
    worst = 0.0
    for b in range(s.batch):
        L = int(w.context_lens[b])
        if L == 0:
            continue
        pos = np.arange(L)
        blk, off = w.block_tables[b][pos // s.block_size], pos % s.block_size
        first_new = max(0, L - q_len)
        for kvh in range(s.num_kv_heads):
            K, V = kc[blk, kvh, off, :].copy(), vc[blk, kvh, off, :].copy()
            K[first_new:] = kn[b, q_len - (L - first_new):, kvh]     # this step's new tokens
            V[first_new:] = vn[b, q_len - (L - first_new):, kvh]
            rows = np.stack([q[b, i, kvh * g + h] for i in range(q_len) for h in range(g)])
            last = np.array([L - q_len + i for i in range(q_len) for _ in range(g)])
            got = _unit_output(rows, K, V, w.scale, last, share)
            x = np.where(pos[None, :] <= last[:, None], rows @ K.T * w.scale, -np.inf)
            seen = np.isfinite(x).any(1)
            e = np.exp(np.where(seen[:, None], x - np.where(seen, x.max(1), 0.0)[:, None], -np.inf))
            den = e.sum(1, keepdims=True)
            ref = (e @ V) / np.where(den > 0, den, 1.0)
            worst = max(worst, float((np.abs(got - ref) / (2e-3 + 1e-2 * np.abs(ref))).max()))
    return worst


EDGE = wl.LLAMA3_8B.replace(name="edge", batch=10, lengths=("fixed", (1, 2, 8, 18, 16, 17, 0, 33, 512, 513)),
                            pool=("factor", 1.5), num_q_heads=8, num_kv_heads=2)       # 32 rows, 16-token steps
SMALL_70B = wl.LLAMA70B_TAIL.replace(name="70b_small", batch=6, lengths=("lognormal", 200.0, 1.0, 1, 900),
                                     shared_prefix=(2, 64))                           # 64 rows, 32-token steps


def test_kernel_constants_were_found():
    assert 0.0 < LO_SHARE < 1.0 and LAZY > 0.0


def test_selective_remainder_keeps_the_error_well_inside_the_bound():
    assert _worst_over_bound(EDGE, 8, 3, LO_SHARE) < 0.5
    assert _worst_over_bound(SMALL_70B, 8, 7, LO_SHARE) < 0.5


def test_weights_without_their_remainder_break_the_bound():
    # One bf16 term per weight (8 significant bits) fails on short contexts
    # whose V values cancel: the remainder is what keeps the rule inside it.
    assert _worst_over_bound(EDGE, 8, 3, None) > 1.0

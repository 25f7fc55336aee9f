"""Pins for the fp64 oracle: checks against things other than the oracle itself.

* brute force: contiguous (unpaged) attention with Python loops, math.exp and
  no max-subtraction, and torch's fp64 scaled_dot_product_attention;
* invariants: block-placement permutation, softmax weights sum to 1, shared
  prefix blocks == private copies, split + log-sum-exp merge == unsplit;
* special cases: one-token context returns V exactly, equal keys give mean(V),
  GQA equals MHA with each KV head repeated g times;
* number formats: every fp16 / bf16 bit pattern against torch's conversion;
  every E4M3 code, and E4M3 rounding of in-range values, against torch's
  float8_e4m3fn; saturation, ties-to-even and subnormals by closed form;
* page worked examples (tests/golden/*.json, each with its source);
* planted mistakes: each mutation of the oracle below is caught by a pin.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def make_contiguous_case(seed, B=3, Hq=8, Hkv=2, D=16, lens=(1, 5, 23), dtype="fp16"):
    """Contiguous per-sequence K/V [B][Hkv][Lmax][D] (bits) + q, as a model would
    hold them before paging."""
    g = torch.Generator().manual_seed(seed)
    tdt = torch.float16 if dtype == "fp16" else torch.bfloat16
    Lmax = max(lens)
    K = torch.randn(B, Hkv, Lmax, D, generator=g).to(tdt)
    V = torch.randn(B, Hkv, Lmax, D, generator=g).to(tdt)
    q = torch.randn(B, Hq, D, generator=g).to(tdt)
    return bits_of(q), bits_of(K), bits_of(V)


def page_it(K_bits, V_bits, lens, block_size, num_blocks, rng):
    """Scatter contiguous K/V into a paged pool with a random block placement;
    unused slots hold NaN so any stray read shows."""
    B, Hkv, _, D = K_bits.shape
    nan_bits = np.uint16(0x7E00)
    kc = np.full((num_blocks, Hkv, block_size, D), nan_bits, np.uint16)
    vc = np.full_like(kc, nan_bits)
    nblk = [-(-L // block_size) for L in lens]
    perm = rng.permutation(num_blocks)
    mb = max(max(nblk), 1)
    tables = np.full((B, mb), -1, np.int32)
    c = 0
    for b, L in enumerate(lens):
        for j in range(nblk[b]):
            tables[b, j] = perm[c]
            c += 1
        for t in range(L):
            blk, off = tables[b, t // block_size], t % block_size
            kc[blk, :, off, :] = K_bits[b, :, t, :]
            vc[blk, :, off, :] = V_bits[b, :, t, :]
    return kc, vc, tables


def brute_force(q_bits, K_bits, V_bits, lens, scale, dtype):
    """Contiguous attention with plain Python loops: exp(s_t) / sum_u exp(s_u)."""
    B, Hq, D = q_bits.shape
    Hkv = K_bits.shape[1]
    g = Hq // Hkv
    q, K, V = (oracle.widen(x, dtype) for x in (q_bits, K_bits, V_bits))
    out = np.zeros((B, Hq, D))
    for b in range(B):
        for h in range(Hq):
            kv = h // g
            L = lens[b]
            if L == 0:
                continue
            s = [scale * math.fsum(q[b, h, d] * K[b, kv, t, d] for d in range(D)) for t in range(L)]
            e = [math.exp(x) for x in s]
            z = math.fsum(e)
            for d in range(D):
                out[b, h, d] = math.fsum(e[t] * V[b, kv, t, d] for t in range(L)) / z
    return out


def sdpa_reference(q_bits, K_bits, V_bits, lens, scale, dtype):
    """torch fp64 scaled_dot_product_attention on each sequence's contiguous K/V."""
    B, Hq, D = q_bits.shape
    Hkv = K_bits.shape[1]
    g = Hq // Hkv
    q, K, V = (torch.from_numpy(oracle.widen(x, dtype)) for x in (q_bits, K_bits, V_bits))
    out = torch.zeros(B, Hq, D, dtype=torch.float64)
    for b in range(B):
        L = lens[b]
        if L == 0:
            continue
        Kb = K[b, :, :L].repeat_interleave(g, dim=0)   # [Hq][L][D]
        Vb = V[b, :, :L].repeat_interleave(g, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(
            q[b][:, None, :], Kb, Vb, scale=scale)
        out[b] = o[:, 0, :]
    return out.numpy()


def paged_case(seed, lens=(1, 5, 23), dtype="fp16", Hq=8, Hkv=2, D=16, bs=4, spare=3):
    q, K, V = make_contiguous_case(seed, B=len(lens), Hq=Hq, Hkv=Hkv, D=D, lens=lens, dtype=dtype)
    nb = sum(-(-L // bs) for L in lens) + spare
    kc, vc, tables = page_it(K, V, lens, bs, nb, np.random.default_rng(seed))
    return q, K, V, kc, vc, tables


# ------------------------------------------------------------------ number formats

def test_widen_fp16_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.widen(bits, "fp16")
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.float16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # closed forms from the binary16 definition
    assert oracle.widen(np.array([0x3C00]), "fp16")[0] == 1.0
    assert oracle.widen(np.array([0xC000]), "fp16")[0] == -2.0
    assert oracle.widen(np.array([0x0001]), "fp16")[0] == 2.0 ** -24
    assert oracle.widen(np.array([0x7BFF]), "fp16")[0] == 65504.0
    assert oracle.widen(np.array([0x7C00]), "fp16")[0] == math.inf


def test_widen_bf16_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.widen(bits, "bf16")
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert oracle.widen(np.array([0x3F80]), "bf16")[0] == 1.0
    assert oracle.widen(np.array([0xC000]), "bf16")[0] == -2.0
    assert oracle.widen(np.array([0x0001]), "bf16")[0] == 2.0 ** -133
    assert oracle.widen(np.array([0x4049]), "bf16")[0] == 3.140625
    assert oracle.widen(np.array([0xFF80]), "bf16")[0] == -math.inf


# ------------------------------------------------------------------ attention vs brute force

@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("seed", [0, 1])
def test_paged_equals_bruteforce_contiguous(seed, dtype):
    lens = (1, 5, 23)
    q, K, V, kc, vc, tables = paged_case(seed, lens=lens, dtype=dtype)
    scale = 1 / math.sqrt(16)
    ours = oracle.decode_attention(q, kc, vc, tables, np.array(lens), scale, dtype, 4)
    bf = brute_force(q, K, V, lens, scale, dtype)
    assert np.abs(ours - bf).max() < 1e-13
    ref = sdpa_reference(q, K, V, lens, scale, dtype)
    assert np.abs(ours - ref).max() < 1e-12


def test_gqa_groups_mha_and_mqa_bruteforce():
    for Hq, Hkv in [(4, 4), (8, 1), (6, 3)]:
        lens = (7, 2)
        q, K, V, kc, vc, tables = paged_case(5, lens=lens, Hq=Hq, Hkv=Hkv, D=8, bs=2)
        ours = oracle.decode_attention(q, kc, vc, tables, np.array(lens), 0.3, "fp16", 2)
        assert np.abs(ours - brute_force(q, K, V, lens, 0.3, "fp16")).max() < 1e-13


def test_scale_is_a_multiplier():
    """scale = 1/sqrt(d) reproduces the listing's scores / sqrt(d_k)."""
    lens = (9,)
    q, K, V, kc, vc, tables = paged_case(3, lens=lens, Hq=2, Hkv=1, D=16)
    ours = oracle.decode_attention(q, kc, vc, tables, np.array(lens), 0.25, "fp16", 4)
    qd, Kd, Vd = (torch.from_numpy(oracle.widen(x, "fp16")) for x in (q, K, V))
    scores = (qd[0] @ Kd[0, 0, :9].T) / math.sqrt(16)
    ref = torch.softmax(scores, dim=-1) @ Vd[0, 0, :9]
    assert np.abs(ours[0] - ref.numpy()).max() < 1e-13


# ------------------------------------------------------------------ invariants

def test_block_placement_permutation_is_invisible():
    lens = (3, 16, 17, 33)
    q, K, V, kc, vc, tables = paged_case(7, lens=lens, spare=6)
    base = oracle.decode_attention(q, kc, vc, tables, np.array(lens), 0.2, "fp16", 4)
    rng = np.random.default_rng(11)
    for _ in range(3):
        perm = rng.permutation(kc.shape[0])           # new home of each block
        kc2 = np.empty_like(kc); vc2 = np.empty_like(vc)
        kc2[perm] = kc; vc2[perm] = vc
        t2 = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
        other = oracle.decode_attention(q, kc2, vc2, t2, np.array(lens), 0.2, "fp16", 4)
        assert np.array_equal(base, other)


def test_softmax_weights_sum_to_one():
    rng = np.random.default_rng(0)
    for L in (1, 2, 17, 1000):
        K = rng.standard_normal((L, 32)); V = rng.standard_normal((L, 32)); q = rng.standard_normal(32)
        _, p, lse = oracle.attend_one(q, K, V, 3.0)
        assert abs(p.sum() - 1.0) < 1e-12
        assert np.all(p >= 0)
        s = 3.0 * K @ q
        assert abs(lse - (s.max() + math.log(np.exp(s - s.max()).sum()))) < 1e-9


def test_one_token_context_returns_v_exactly():
    lens = (1, 1)
    q, K, V, kc, vc, tables = paged_case(2, lens=lens)
    out = oracle.decode_attention(q, kc, vc, tables, np.array(lens), 0.7, "fp16", 4)
    Vd = oracle.widen(V, "fp16")
    for b in range(2):
        for h in range(8):
            assert np.array_equal(out[b, h], Vd[b, h // 4, 0])


def test_equal_keys_give_mean_of_v():
    q, K, V, kc, vc, tables = paged_case(4, lens=(37,))
    kc[:] = kc[tables[0, 0], :, 0:1, :]  # every slot gets the same key
    out = oracle.decode_attention(q, kc, vc, tables, np.array([37]), 0.5, "fp16", 4)
    Vd = oracle.widen(V, "fp16")
    for h in range(8):
        assert np.abs(out[0, h] - Vd[0, h // 4, :37].mean(axis=0)).max() < 1e-12


def test_gqa_equals_mha_with_repeated_kv_heads():
    lens = (6, 19)
    q, K, V, kc, vc, tables = paged_case(8, lens=lens, Hq=8, Hkv=2)
    gqa = oracle.decode_attention(q, kc, vc, tables, np.array(lens), 0.3, "fp16", 4)
    mha = oracle.decode_attention(q, np.repeat(kc, 4, axis=1), np.repeat(vc, 4, axis=1),
                                  tables, np.array(lens), 0.3, "fp16", 4)
    assert np.array_equal(gqa, mha)


def test_split_merge_identity():
    rng = np.random.default_rng(1)
    for L, split in [(1, 4), (33, 8), (100, 7), (512, 512), (513, 512)]:
        K = rng.standard_normal((L, 16)); V = rng.standard_normal((L, 16)); q = rng.standard_normal(16)
        whole = oracle.attend_one(q, K, V, 0.9)[0]
        merged = oracle.lse_merge(oracle.split_partials(q, K, V, 0.9, split))
        assert np.abs(whole - merged).max() < 1e-12
    # an empty split carries zero weight
    parts = [(np.ones(4), 0.5), (np.zeros(4), -math.inf)]
    assert np.array_equal(oracle.lse_merge(parts), np.ones(4))


def test_shared_prefix_equals_private_copies():
    bs = 4
    q, K, V = make_contiguous_case(9, B=3, lens=(13, 13, 13))
    K[1, :, :8] = K[0, :, :8]; V[1, :, :8] = V[0, :, :8]   # 8-token shared prefix
    K[2, :, :8] = K[0, :, :8]; V[2, :, :8] = V[0, :, :8]
    kc, vc, private = page_it(K, V, (13, 13, 13), bs, 16, np.random.default_rng(0))
    shared = private.copy()
    shared[1, :2] = private[0, :2]
    shared[2, :2] = private[0, :2]
    a = oracle.decode_attention(q, kc, vc, private, np.array([13] * 3), 0.25, "fp16", bs)
    b = oracle.decode_attention(q, kc, vc, shared, np.array([13] * 3), 0.25, "fp16", bs)
    assert np.array_equal(a, b)


def test_empty_context_gives_zeros():
    q, K, V, kc, vc, tables = paged_case(1, lens=(0, 3))
    out = oracle.decode_attention(q, kc, vc, tables, np.array([0, 3]), 0.25, "fp16", 4)
    assert np.array_equal(out[0], np.zeros_like(out[0]))
    assert np.all(np.isfinite(out))


# ------------------------------------------------------------------ append

def test_append_is_a_byte_permutation_and_matches_torch_cat():
    """Appending token L-1 through the slot mapping, then attending, equals
    torch.cat of the new K/V onto contiguous K/V (the pre-paging cache)."""
    lens_before = (0, 4, 15, 16)
    bs, Hq, Hkv, D = 4, 4, 2, 8
    lens = tuple(L + 1 for L in lens_before)
    q, K, V = make_contiguous_case(12, B=4, Hq=Hq, Hkv=Hkv, D=D, lens=lens)
    nan = np.uint16(0x7E00)
    Kold = K.copy(); Vold = V.copy()
    for b, L in enumerate(lens_before):
        Kold[b, :, L:] = nan; Vold[b, :, L:] = nan
    kc, vc, tables = page_it(Kold, Vold, lens, bs, 12, np.random.default_rng(3))
    slots = oracle.slot_mapping(tables, np.array(lens), bs)
    k_new = np.stack([K[b, :, L] for b, L in enumerate(lens_before)])
    v_new = np.stack([V[b, :, L] for b, L in enumerate(lens_before)])
    kc2, vc2 = oracle.kv_append(kc, vc, k_new, v_new, slots, bs)
    changed = np.argwhere(np.any(kc2 != kc, axis=(1, 3)))
    assert sorted(map(tuple, changed)) == sorted((int(s) // bs, int(s) % bs) for s in slots)
    out = oracle.decode_attention(q, kc2, vc2, tables, np.array(lens), 0.3, "fp16", bs)
    assert np.abs(out - brute_force(q, K, V, lens, 0.3, "fp16")).max() < 1e-13
    # negative slot -> nothing stored
    kc3, _ = oracle.kv_append(kc, vc, k_new, v_new, np.full(4, -1, np.int32), bs)
    assert np.array_equal(kc3, kc)


def test_slot_mapping_on_page_block_tables(golden_dir):
    gold = json.load(open(os.path.join(golden_dir, "block_tables.json")))
    bs = gold["block_size"]
    for page in ("kasblo", "youngju"):
        for req, table in gold[page]["tables"].items():
            row = np.array(table, np.int32)
            for pos, slot in zip(gold[page]["positions"][req], gold[page]["slots"][req]):
                assert oracle.slot_of_position(row, pos, bs) == slot
    tables = np.array([[7, 1, 9], [3, 8, -1]], np.int32)
    assert list(oracle.slot_mapping(tables, np.array([48, 20]), bs)) == [159, 131]
    assert list(oracle.slot_mapping(tables, np.array([0, 1]), bs)) == [-1, 48]


# ------------------------------------------------------------------ accounting vs the pages

def test_kv_accounting_worked_examples(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "kv_accounting.json")))
    w = g["kasblo_worked_example"]
    m = oracle.kv_bytes_per_token(w["layers"], w["kv_heads"], w["head_dim"], w["elem_bytes"])
    assert m == w["m_token_bytes"]
    assert w["block_size"] * m == w["block_bytes"]
    assert oracle.blocks_needed(w["tokens"], w["block_size"]) == w["n_blocks"]
    assert w["tokens"] * m == w["token_bytes_formula"]
    assert oracle.allocated_bytes(w["tokens"], w["block_size"], m) == w["alloc_bytes_formula"]
    assert oracle.wasted_bytes(w["tokens"], w["block_size"], m) == w["waste_bytes_formula"]
    # the page's table used the block size where the token size belongs (x16)
    printed = w["printed_table_mib"]
    mib = 2 ** 20
    assert printed["tokens"] * mib == w["block_size"] * w["token_bytes_formula"]
    assert printed["allocated"] * mib == w["block_size"] * w["alloc_bytes_formula"]
    assert printed["unused_tail"] * mib == w["block_size"] * w["waste_bytes_formula"]
    b = g["babushkai_llama3_70b"]
    m70 = oracle.kv_bytes_per_token(b["layers"], b["kv_heads"], b["head_dim"], b["elem_bytes"])
    assert m70 == b["m_token_kib"] * 1024
    assert m70 * b["context_tokens"] == b["total_gib"] * 2 ** 30
    s = g["scalingbook_llama2_13b"]
    tot = oracle.kv_cache_bytes(s["tokens"], s["layers"], s["kv_heads"], s["head_dim"], 1, s["elem_bytes"])
    assert round(tot / 1e9, 1) == s["approx_gb"]
    # waste stays below one block for every length
    for n in range(1, 200):
        assert 0 <= oracle.wasted_bytes(n, 16, 1) < 16


def test_roofline_step_time_printed_values(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "step_time.json")))
    for batch, (total, per_stream) in g["printed"].items():
        tps = oracle.decode_step_tokens_per_s(int(batch), g["ctx"], g["bandwidth"], g["compute"],
                                              g["weight_bytes"], g["kv_bytes_per_token"], g["params"])
        assert round(tps) == total
        assert round(tps / int(batch), 1) == per_stream
    ceiling = oracle.decode_step_tokens_per_s(1, 0, g["bandwidth"], g["compute"], g["weight_bytes"], 0, g["params"])
    assert round(ceiling) == g["single_stream_ceiling_tok_s"]


def test_attention_bytes_formula():
    # 2 sequences of 10 and 6 tokens, Hkv=2, D=4, 2-byte values, Hq=4, 3 table entries read
    n = oracle.attention_call_bytes([10, 6], 2, 4, 2, 4, 2, 3)
    assert n == 16 * 2 * 4 * 2 * 2 + 2 * 2 * 4 * 4 * 2 + 12 + 8


# ------------------------------------------------------------------ planted mistakes

def _pins_pass():
    """The brute-force and placement pins, as a function of the current oracle."""
    lens = (1, 5, 23)
    q, K, V, kc, vc, tables = paged_case(0, lens=lens)
    ours = oracle.decode_attention(q, kc, vc, tables, np.array(lens), 0.25, "fp16", 4)
    return np.all(np.isfinite(ours)) and np.abs(ours - brute_force(q, K, V, lens, 0.25, "fp16")).max() < 1e-13


MUTATIONS = {
    "kv head h % Hkv": ("kv_head_of", lambda h, g: h % 2),
    "offset reversed in block": ("gather_kv", lambda c, row, L, kv, bs: c[np.asarray(row, np.int64)[np.arange(L) // bs], kv, bs - 1 - np.arange(L) % bs, :]),
    "logical block not translated": ("gather_kv", lambda c, row, L, kv, bs: c[np.arange(L) // bs, kv, np.arange(L) % bs, :]),
    "scale dropped": ("attend_one", lambda q, K, V, s, f=oracle.attend_one: f(q, K, V, 1.0)),
    "last token dropped": ("gather_kv", lambda c, row, L, kv, bs, f=oracle.gather_kv: f(c, row, max(L - 1, 1), kv, bs)),
    "K and V swapped": ("attend_one", lambda q, K, V, s, f=oracle.attend_one: f(q, V, K, s)),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(monkeypatch, name):
    assert _pins_pass()
    attr, bad = MUTATIONS[name]
    monkeypatch.setattr(oracle, attr, bad)
    assert not _pins_pass()


# ------------------------------------------------------------------ fp8 (E4M3) codes

def test_e4m3_decode_every_code_against_torch_and_closed_forms():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan) and nan.sum() == 2        # 0x7F, 0xFF
    assert np.array_equal(ours[~nan], ref[~nan])
    assert oracle.e4m3_decode(np.array([0x38]))[0] == 1.0                # 0.0111.000
    assert oracle.e4m3_decode(np.array([0x7E]))[0] == 448.0              # largest finite
    assert oracle.e4m3_decode(np.array([0x01]))[0] == 2.0 ** -9          # smallest subnormal
    assert oracle.e4m3_decode(np.array([0x08]))[0] == 2.0 ** -6          # smallest normal
    assert oracle.e4m3_decode(np.array([0xC4]))[0] == -3.0               # 1.1000.100


def test_e4m3_encode_round_trip_ties_and_saturation():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_decode(codes)
    # every finite code encodes back to itself (-0 and +0 both map to their own codes)
    assert np.array_equal(oracle.e4m3_encode(vals.astype(np.float32)), codes)
    # midpoints between neighbours round to the even mantissa
    pos = np.sort(vals[vals > 0])
    mids = (pos[:-1] + pos[1:]) / 2
    got = oracle.e4m3_decode(oracle.e4m3_encode(mids.astype(np.float32)))
    even = np.where(oracle.e4m3_encode(pos[:-1].astype(np.float32)) % 2 == 0, pos[:-1], pos[1:])
    assert np.array_equal(got, even)
    # saturation instead of overflow, NaN stays NaN, 2^-10 (half the smallest step) rounds to 0
    assert list(oracle.e4m3_encode(np.array([449.0, 464.0, 1e9, -1e9, np.inf], np.float32))) == [0x7E, 0x7E, 0x7E, 0xFE, 0x7E]
    assert oracle.e4m3_encode(np.array([np.nan], np.float32))[0] == 0x7F
    assert oracle.e4m3_encode(np.array([2.0 ** -10], np.float32))[0] == 0


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-12, 6, 200000))).astype(np.float32)
    x = x[np.abs(x) < 448]
    ours = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_quantize_divides_in_float32_then_rounds():
    bits = torch.tensor([1.0, -2.5, 300.0, 0.0078125, 1000.0], dtype=torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    codes = oracle.quantize_e4m3(bits, "bf16", 0.5)
    assert list(oracle.e4m3_decode(codes)) == [2.0, -5.0, 448.0, 0.015625, 448.0]   # 600, 2000 saturate
    # the scale's float32 rounding is what the division sees
    bits1 = torch.tensor([3.0], dtype=torch.float16).view(torch.int16).numpy().view(np.uint16)
    s = 0.1  # not exact in float32
    y = np.float32(3.0) / np.float32(s)
    assert oracle.quantize_e4m3(bits1, "fp16", s)[0] == oracle.e4m3_encode(np.array([y]))[0]


def test_fp8_attention_is_attention_on_dequantised_values():
    lens = (5, 23)
    q, K, V, kc, vc, tables = paged_case(13, lens=lens, dtype="bf16")
    ks, vs = np.array([0.05, 0.03], np.float32), np.array([0.02, 0.04], np.float32)
    kq = np.stack([oracle.quantize_e4m3(kc[:, h], "bf16", ks[h]) for h in range(2)], axis=1)
    vq = np.stack([oracle.quantize_e4m3(vc[:, h], "bf16", vs[h]) for h in range(2)], axis=1)
    rows = [(b, h) for b in range(2) for h in range(8)]
    out = oracle.decode_attention_rows(q, kq, vq, tables, np.array(lens), 0.25, "bf16", 4, rows, kv_scales=(ks, vs))
    # the same attention on the dequantised contiguous arrays, by brute force;
    # the codes are decoded by torch's float8_e4m3fn and multiplied by the
    # float32 scale here, not by the oracle's dequantisation
    Kd = np.stack([_torch_dequant(oracle.quantize_e4m3(K[:, h], "bf16", ks[h]), ks[h]) for h in range(2)], 1)
    Vd = np.stack([_torch_dequant(oracle.quantize_e4m3(V[:, h], "bf16", vs[h]), vs[h]) for h in range(2)], 1)
    qd = oracle.widen(q, "bf16")
    for i, (b, h) in enumerate(rows):
        s = [0.25 * float(qd[b, h] @ Kd[b, h // 4, t]) for t in range(lens[b])]
        e = np.exp(np.array(s) - max(s))
        ref = (e[:, None] * Vd[b, h // 4, :lens[b]]).sum(0) / e.sum()
        assert np.abs(out[i] - ref).max() < 1e-12
    # each code is within half a grid step of the float32 quotient x / scale
    # (the quotient is rounded to float32 first, so ties are decided there)
    x = oracle.widen(K, "bf16").astype(np.float32)
    for h in range(2):
        y = (x[:, h] / ks[h]).astype(np.float64)
        c = oracle.e4m3_decode(oracle.quantize_e4m3(K[:, h], "bf16", ks[h]))
        half = 0.5 * 2.0 ** (np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -6))) - 3)
        assert np.all(np.abs(c - y) <= half)


def _torch_dequant(codes, scale):
    """value = code's E4M3 value (torch's float8_e4m3fn decoding) x float32(scale)."""
    v = torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return v * float(np.float32(scale))


def _torch_quant(x_f32, scale):
    """E4M3 code of float32(x) / float32(scale) by torch: the float32 quotient,
    clamped to +-448 (saturation), then torch's float8_e4m3fn rounding."""
    y = torch.from_numpy(np.asarray(x_f32, np.float32)) / torch.tensor(np.float32(scale))
    return y.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _dequant_pins_pass():
    """dequantize_e4m3 against closed forms: value = E4M3(code) x scale, with
    the scale as the float32 the library stores (design.babushkai.com
    "GPU推論の内部構造", section "KVキャッシュの台帳": FP8 codes with a scale)."""
    for s in (1.0, 0.25, 0.1, 0.0137, 3.5):
        s32 = float(np.float32(s))
        d = oracle.dequantize_e4m3
        checks = [
            (0x38, s32),                 # 0.0111.000 = 1
            (0x7E, 448.0 * s32),         # 0.1111.110 = largest finite
            (0xB8, -s32),                # sign bit
            (0x40, 2.0 * s32),           # 0.1000.000 = 2
            (0x30, 0.5 * s32),           # 0.0110.000 = 1/2
            (0x3C, 1.5 * s32),           # 0.0111.100 = 1 + 4/8
        ]
        checks += [(k, k * 2.0 ** -9 * s32) for k in range(1, 8)]       # subnormals k 2^-9
        checks += [(0x80 | k, -k * 2.0 ** -9 * s32) for k in range(1, 8)]
        for code, want in checks:
            if d(np.array([code], np.uint8), s)[0] != want:
                return False
        if d(np.array([0x00], np.uint8), s)[0] != 0.0 or not np.isnan(d(np.array([0x7F], np.uint8), s)[0]):
            return False
    return True


def test_dequantize_closed_forms():
    assert _dequant_pins_pass()


def test_dequantize_equals_torch_decode_times_float32_scale():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    for s in (0.004, 0.0199, 0.1, 1.0, 7.25):
        assert np.array_equal(oracle.dequantize_e4m3(codes, s), _torch_dequant(codes, s))


def test_quantize_then_dequantize_within_half_a_step():
    """|dequantize(quantize(x, s), s) - x| <= s * (half the E4M3 spacing at
    x / s) + |x| 2^-23 (the float32 rounding of the quotient), for |x / s| <= 448."""
    g = torch.Generator().manual_seed(5)
    for s in (0.004, 0.02, 0.3):
        x = (torch.randn(50000, generator=g) * 3.0).to(torch.bfloat16)
        xb = bits_of(x)
        xv = oracle.widen(xb, "bf16")
        keep = np.abs(xv / s) <= 440.0
        got = oracle.dequantize_e4m3(oracle.quantize_e4m3(xb, "bf16", s), s)
        y = np.abs(xv / float(np.float32(s)))
        half = 0.5 * 2.0 ** (np.floor(np.log2(np.maximum(y, 2.0 ** -6))) - 3)
        bound = float(np.float32(s)) * half + np.abs(xv) * 2.0 ** -23
        assert np.all(np.abs(got - xv)[keep] <= bound[keep])
        # and outside the range the value saturates at +-448 s
        big = np.abs(xv / s) > 470.0
        if big.any():
            assert np.all(np.abs(got[big]) == 448.0 * float(np.float32(s)))


def _fp8_append_case():
    """Two KV heads whose K and V scales differ by orders of magnitude, three
    tokens (one skipped) in a pool of 3 blocks of 4 slots."""
    g = torch.Generator().manual_seed(11)
    kn = (torch.randn(3, 2, 16, generator=g) * torch.tensor([0.5, 40.0]).view(1, 2, 1)).to(torch.bfloat16)
    vn = (torch.randn(3, 2, 16, generator=g) * torch.tensor([20.0, 0.02]).view(1, 2, 1)).to(torch.bfloat16)
    ks = np.array([0.003, 0.25], np.float32)
    vs = np.array([0.09, 0.0001], np.float32)
    slots = np.array([9, -1, 2], np.int32)
    kc = np.full((3, 2, 4, 16), 0x7F, np.uint8)
    vc = np.full((3, 2, 4, 16), 0x7F, np.uint8)
    return kn, vn, ks, vs, slots, kc, vc


def _fp8_append_pin_passes():
    """kv_append_fp8 against codes built by torch: token i, KV head h holds
    E4M3(float32(k) / k_scale[h]) in k_cache[slot // 4][h][slot % 4] and
    E4M3(float32(v) / v_scale[h]) in v_cache likewise; other slots keep their
    bytes."""
    kn, vn, ks, vs, slots, kc, vc = _fp8_append_case()
    k_out, v_out = oracle.kv_append_fp8(kc, vc, bits_of(kn), bits_of(vn), slots, 4, ks, vs, "bf16")
    k_want, v_want = kc.copy(), vc.copy()
    for i, slot in enumerate(slots):
        if slot < 0:
            continue
        for h in range(2):
            k_want[slot // 4, h, slot % 4] = _torch_quant(kn[i, h].float().numpy(), ks[h])
            v_want[slot // 4, h, slot % 4] = _torch_quant(vn[i, h].float().numpy(), vs[h])
    return np.array_equal(k_out, k_want) and np.array_equal(v_out, v_want)


def test_fp8_append_uses_each_heads_own_k_and_v_scale():
    assert _fp8_append_pin_passes()
    kn, vn, ks, vs, slots, kc, vc = _fp8_append_case()
    k_out, _ = oracle.kv_append_fp8(kc, vc, bits_of(kn), bits_of(vn), slots, 4, ks, vs, "bf16")
    # the values really do depend on the scale chosen: head 0's K with head 1's scale differs
    assert not np.array_equal(k_out[2, 0, 1], _torch_quant(kn[0, 0].float().numpy(), ks[1]))
    # untouched slots keep the NaN code
    assert np.all(k_out[0, :, 0] == 0x7F) and np.all(k_out[1] == 0x7F)


def _fp8_pins_pass():
    """The E4M3 pins above, as a function of the current oracle."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = oracle.e4m3_decode(codes)
    if not (np.array_equal(np.isnan(ours), np.isnan(ref)) and np.array_equal(ours[~np.isnan(ref)], ref[~np.isnan(ref)])):
        return False
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-12, 6, 20000))).astype(np.float32)
    x = x[np.abs(x) < 448]
    if not np.array_equal(oracle.e4m3_encode(x), torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()):
        return False
    if list(oracle.e4m3_encode(np.array([1e9, -1e9], np.float32))) != [0x7E, 0xFE]:
        return False
    return _dequant_pins_pass() and _fp8_append_pin_passes()


def _truncating_encode(x, f=oracle.e4m3_encode):
    """Rounds toward zero instead of to nearest."""
    x = np.asarray(x, np.float32)
    c = f(x)
    over = np.abs(oracle.e4m3_decode(c)) > np.abs(x.astype(np.float64))
    return np.where(over & (c & 0x7F > 0), c - 1, c).astype(np.uint8)


FP8_MUTATIONS = {
    "exponent bias 8": ("e4m3_decode", lambda c, f=oracle.e4m3_decode: f(c) / 2.0),
    "no saturation": ("e4m3_encode", lambda x, f=oracle.e4m3_encode: np.where(np.abs(np.asarray(x, np.float32)) > 448, 0x7F, f(x)).astype(np.uint8)),
    "round toward zero": ("e4m3_encode", _truncating_encode),
    "subnormals flushed": ("e4m3_decode", lambda c, f=oracle.e4m3_decode: np.where((np.asarray(c) & 0x78) == 0, 0.0, f(c))),
    "dequantise by division": ("dequantize_e4m3", lambda c, s, f=oracle.e4m3_decode: f(c) / float(np.float32(s))),
    "dequantise with a float64 scale": ("dequantize_e4m3", lambda c, s, f=oracle.e4m3_decode: f(c) * float(s)),
    "append: K and V scales swapped": (
        "kv_append_fp8", lambda kc, vc, kn, vn, sl, bs, ks, vs, dt, f=oracle.kv_append_fp8: f(kc, vc, kn, vn, sl, bs, vs, ks, dt)),
    "append: KV head index off by one": (
        "kv_append_fp8", lambda kc, vc, kn, vn, sl, bs, ks, vs, dt, f=oracle.kv_append_fp8:
        f(kc, vc, kn, vn, sl, bs, np.roll(ks, 1), np.roll(vs, 1), dt)),
    "append: quantise by multiplication": (
        "quantize_e4m3", lambda b, dt, s, f=oracle.quantize_e4m3: f(b, dt, 1.0 / float(s))),
}


@pytest.mark.parametrize("name", sorted(FP8_MUTATIONS))
def test_planted_fp8_mistake_is_caught(monkeypatch, name):
    assert _fp8_pins_pass()
    attr, bad = FP8_MUTATIONS[name]
    monkeypatch.setattr(oracle, attr, bad)
    assert not _fp8_pins_pass()


# ------------------------------------------------------------------ several new tokens per sequence

def _causal_bruteforce(q_bits, K_bits, V_bits, lens, q_len, scale, dtype):
    """Contiguous causal attention with Python loops: new token i of sequence
    b (position L - q_len + i) against keys 0 .. L - q_len + i."""
    B, n, Hq, D = q_bits.shape
    g = Hq // K_bits.shape[1]
    q, K, V = (oracle.widen(x, dtype) for x in (q_bits, K_bits, V_bits))
    out = np.zeros((B, n, Hq, D))
    for b in range(B):
        for i in range(n):
            pos = lens[b] - n + i
            if pos < 0:
                continue
            for h in range(Hq):
                s = [scale * math.fsum(q[b, i, h, d] * K[b, h // g, t, d] for d in range(D)) for t in range(pos + 1)]
                e = [math.exp(x) for x in s]
                z = math.fsum(e)
                for d in range(D):
                    out[b, i, h, d] = math.fsum(e[t] * V[b, h // g, t, d] for t in range(pos + 1)) / z
    return out


def _multi_case(seed, lens, n, Hq=4, Hkv=2, D=8, bs=4):
    q1, K, V, kc, vc, tables = paged_case(seed, lens=lens, Hq=Hq, Hkv=Hkv, D=D, bs=bs)
    g = torch.Generator().manual_seed(seed + 100)
    q = bits_of(torch.randn(len(lens), n, Hq, D, generator=g).to(torch.float16))
    return q, K, V, kc, vc, tables


@pytest.mark.parametrize("n", [1, 2, 3, 5])
def test_multi_query_equals_causal_bruteforce(n):
    lens = (7, 2, 13, 0)
    q, K, V, kc, vc, tables = _multi_case(4, lens, n)
    ours = oracle.decode_attention_multi(q, kc, vc, tables, np.array(lens), n, 0.4, "fp16", 4)
    ref = _causal_bruteforce(q, K, V, lens, n, 0.4, "fp16")
    assert np.abs(ours - ref).max() < 1e-13
    # a sequence shorter than q_len: its first tokens have no keys and give zero rows
    assert np.all(ours[1, :max(0, n - 2)] == 0)


def test_multi_query_rows_are_single_token_decodes_of_the_prefix():
    """New token i is exactly a one-token decode with context L - q_len + i + 1."""
    lens, n = (9, 16, 17), 4
    q, K, V, kc, vc, tables = _multi_case(6, lens, n)
    ours = oracle.decode_attention_multi(q, kc, vc, tables, np.array(lens), n, 0.3, "fp16", 4)
    for i in range(n):
        ctx = np.array([L - n + i + 1 for L in lens])
        one = oracle.decode_attention(q[:, i], kc, vc, tables, ctx, 0.3, "fp16", 4)
        assert np.array_equal(ours[:, i], one)
    # q_len = 1 is the one-token decode itself
    q1 = q[:, :1]
    assert np.array_equal(oracle.decode_attention_multi(q1, kc, vc, tables, np.array(lens), 1, 0.3, "fp16", 4)[:, 0],
                          oracle.decode_attention(q1[:, 0], kc, vc, tables, np.array(lens), 0.3, "fp16", 4))


def test_slot_mapping_multi_on_page_block_tables(golden_dir):
    gold = json.load(open(os.path.join(golden_dir, "block_tables.json")))
    bs = gold["block_size"]
    A = gold["kasblo"]
    table = np.array([A["tables"]["A"]], np.int32)
    printed = dict(zip(A["positions"]["A"], A["slots"]["A"]))
    # L = 33 with 3 new tokens: positions 30, 31, 32 (31 and 32 printed on the page: 31, 144)
    slots = oracle.slot_mapping_multi(table, np.array([33]), 3, bs)[0]
    assert slots[1] == printed[31] and slots[2] == printed[32] and slots[0] == printed[31] - 1
    # L = 17 with 2 new tokens: positions 15, 16 -> 127, 16
    assert list(oracle.slot_mapping_multi(table, np.array([17]), 2, bs)[0]) == [printed[15], printed[16]]
    # fewer tokens than new tokens: the missing positions are -1
    assert list(oracle.slot_mapping_multi(table, np.array([1]), 3, bs)[0]) == [-1, -1, printed[0]]


def _bad_multi(q_bits, kc, vc, tables, lens, n, scale, dtype, bs, kv_scales=None, rows=None,
               f=oracle.decode_attention_multi):
    """Off by one in the causal limit: token i also sees token i + 1."""
    return f(q_bits, kc, vc, tables, np.asarray(lens) + 1, n, scale, dtype, bs, kv_scales, rows)


def test_planted_causal_off_by_one_is_caught(monkeypatch):
    lens, n = (7, 13), 3
    q, K, V, kc, vc, tables = _multi_case(2, lens, n)
    ref = _causal_bruteforce(q, K, V, lens, n, 0.4, "fp16")
    good = oracle.decode_attention_multi(q, kc, vc, tables, np.array(lens), n, 0.4, "fp16", 4)
    assert np.abs(good - ref).max() < 1e-13
    monkeypatch.setattr(oracle, "decode_attention_multi", _bad_multi)
    bad = oracle.decode_attention_multi(q, kc, vc, tables, np.array(lens), n, 0.4, "fp16", 4)
    assert not np.abs(bad - ref).max() < 1e-13


# ------------------------------------------------------------------ copy-on-write

def test_copy_blocks_is_a_block_permutation_of_bytes():
    rng = np.random.default_rng(3)
    kc = rng.integers(0, 2 ** 16, size=(9, 2, 4, 8), dtype=np.uint16)
    vc = rng.integers(0, 2 ** 16, size=(9, 2, 4, 8), dtype=np.uint16)
    pairs = [(1, 5), (3, 7), (1, 8)]
    k, v = oracle.copy_blocks(kc, vc, pairs)
    for src, dst in pairs:
        assert np.array_equal(k[dst], kc[src]) and np.array_equal(v[dst], vc[src])
    untouched = [b for b in range(9) if b not in (5, 7, 8)]
    assert np.array_equal(k[untouched], kc[untouched]) and np.array_equal(v[untouched], vc[untouched])
    assert np.array_equal(oracle.copy_blocks(kc, vc, [])[0], kc)


def test_forked_sequences_see_the_prefix_and_their_own_tokens_after_copy_on_write():
    """Two sequences share a 6-token prefix (block size 4: one full and one
    partial block).  Each then writes its own tokens: the copy of the partial
    block before the first write keeps the prefix for both, and neither sees
    the other's tokens."""
    bs, D = 4, 8
    kc = np.full((6, 1, bs, D), 0x7E00, np.uint16)
    vc = kc.copy()
    rng = np.random.default_rng(0)
    prefix = rng.integers(0, 0x3C00, size=(6, D), dtype=np.uint16)
    table_a = [2, 4]                       # the prefix: block 2 full, block 4 holds tokens 4, 5
    for t in range(6):
        kc[table_a[t // bs], 0, t % bs] = prefix[t]
        vc[table_a[t // bs], 0, t % bs] = prefix[t] ^ 1
    table_b = list(table_a)                # the fork shares both blocks
    kc, vc = oracle.copy_blocks(kc, vc, [(4, 1)])   # b writes position 6 into shared block 4: copy it first
    table_b[1] = 1
    own_a = rng.integers(0, 0x3C00, size=(3, D), dtype=np.uint16)
    own_b = rng.integers(0, 0x3C00, size=(3, D), dtype=np.uint16)
    table_a.append(0)
    table_b.append(3)
    for i in range(3):
        pos = 6 + i
        kc, vc = oracle.kv_append(kc, vc, own_a[i:i + 1, None], own_a[i:i + 1, None] ^ 1,
                                  np.array([table_a[pos // bs] * bs + pos % bs]), bs)
        kc, vc = oracle.kv_append(kc, vc, own_b[i:i + 1, None], own_b[i:i + 1, None] ^ 1,
                                  np.array([table_b[pos // bs] * bs + pos % bs]), bs)
    ka = oracle.gather_kv(kc, np.array(table_a), 9, 0, bs)
    kb = oracle.gather_kv(kc, np.array(table_b), 9, 0, bs)
    assert np.array_equal(ka, np.concatenate([prefix, own_a])) and np.array_equal(kb, np.concatenate([prefix, own_b]))
    assert np.array_equal(oracle.gather_kv(vc, np.array(table_b), 9, 0, bs), np.concatenate([prefix, own_b]) ^ 1)

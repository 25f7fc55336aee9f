"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Append: bit-exact over the whole pool, untouched (NaN-sentinel) slots included.
Attention: |gpu - ref| <= 2e-3 + 1e-2 |ref| elementwise, ref in float64 from
the same rounded inputs.  Small cases compare every output; the full-size
configurations use the launch configuration the bench times (automatic
splits) and compare every output where the oracle finishes in seconds,
otherwise seeded samples of (sequence, query head) rows.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_26_gb300 as pkv
import workloads as wl
from paged_kv_cache_26_gb300 import build as pkv_build
from parity_helpers import (ATOL, RTOL, assert_close, bits, oracle_all_rows, oracle_caches, oracle_rows,
                            run_gpu_step, sample_rows, widen_out)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv_build.build()


def full_check(w, num_splits, layer=0, rows=None, fused=False):
    out, kc, vc = run_gpu_step(w, layer, num_splits, fused=fused)
    rk, rv = oracle_caches(w, layer)
    assert np.array_equal(bits(kc), rk), "K append differs from the oracle"
    assert np.array_equal(bits(vc), rv), "V append differs from the oracle"
    B, H, D = w.spec.batch, w.spec.num_q_heads, w.spec.head_dim
    gpu = widen_out(out, w.spec.dtype)
    if rows is None:
        rows = [(b, h) for b in range(B) for h in range(H)]
    ref = oracle_rows(w, rk, rv, rows, layer)
    got = np.stack([gpu[b, h] for b, h in rows])
    assert_close(got, ref, f"{w.spec.name} splits={num_splits} fused={fused}")
    return out


# ---------------------------------------------------------------- the configurations

@pytest.mark.parametrize("splits", [1, 0, 2, 3, 7])
def test_tiny_config_every_output(splits):
    full_check(wl.generate(wl.TINY, seed=0), splits)


REDUCED = [
    wl.LLAMA3_8B.replace(name="llama8b_small", batch=6, lengths=("uniform", 1, 700)),
    wl.MHA_7B_B16.replace(name="mha_small", batch=3, lengths=("constant", 333), num_layers=2),
    wl.LLAMA70B_TAIL.replace(name="70b_small", batch=24, lengths=("lognormal", 200.0, 1.0, 1, 900),
                             shared_prefix=(4, 64)),
    wl.LONG_CTX.replace(name="long_small", batch=2, lengths=("constant", 2100)),
    wl.TINY.replace(name="tiny_bf16_mqa", num_q_heads=8, num_kv_heads=1, dtype="bf16", pool=("factor", 2.0)),
    wl.TINY.replace(name="tiny_d128_g2", num_q_heads=4, num_kv_heads=2, head_dim=128, pool=("factor", 1.5)),
]


@pytest.mark.parametrize("splits", [1, 0, 5])
@pytest.mark.parametrize("spec", REDUCED, ids=lambda s: s.name)
def test_reduced_configs_every_output(spec, splits):
    w = wl.generate(spec, seed=3)
    for layer in range(len(w.q)):
        full_check(w, splits, layer)


def test_llama3_8b_full_every_output():
    w = wl.generate(wl.LLAMA3_8B, seed=0, device="cuda")
    full_check(w, 0)


def test_llama3_8b_full_single_pass_sampled():
    w = wl.generate(wl.LLAMA3_8B, seed=1, device="cuda")
    full_check(w, 1, rows=sample_rows(w, 64))


def full_check_every_output(w, num_splits, layer=0):
    """full_check over every output row, with the oracle gathering each
    (sequence, KV head) once."""
    out, kc, vc = run_gpu_step(w, layer, num_splits)
    rk, rv = oracle_caches(w, layer)
    assert np.array_equal(bits(kc), rk), "K append differs from the oracle"
    assert np.array_equal(bits(vc), rv), "V append differs from the oracle"
    assert_close(widen_out(out, w.spec.dtype), oracle_all_rows(w, rk, rv, layer),
                 f"{w.spec.name} splits={num_splits} layer={layer}")
    return out


def test_llama70b_tail_full_every_output():
    # 256 sequences x 64 query heads, lognormal lengths, 64 sequences sharing a
    # 512-token prefix: every output row against the oracle.
    w = wl.generate(wl.LLAMA70B_TAIL, seed=0, device="cuda")
    assert w.shared_seqs.size == 64
    full_check_every_output(w, 0)


def test_mha7b_b16_full_sampled():
    # Every layer is an identical, independent call; two layers are checked.
    w = wl.generate(wl.MHA_7B_B16, seed=0, device="cuda", layers=2)
    for layer in range(2):
        full_check(w, 0, layer, rows=sample_rows(w, 48, seed=layer))


def test_mha7b_b64_eight_of_32_layers_sampled():
    # Batch 64 x 4096 tokens, 32 query / 32 KV heads: 8 of the configuration's
    # 32 layer calls (each its own cache, the same tables), 96 seeded rows each.
    w = wl.generate(wl.MHA_7B_B64, seed=0, device="cuda", layers=8)
    for layer in range(8):
        full_check(w, 0, layer, rows=sample_rows(w, 96, seed=layer))


@pytest.mark.parametrize("splits", [64, 0])
def test_long_context_split_k_full_every_output(splits):
    # 8 sequences x 32768 tokens with one +8-logit spike key each: all 256 rows.
    w = wl.generate(wl.LONG_CTX, seed=0, device="cuda")
    full_check_every_output(w, splits)


# ---------------------------------------------------------------- edge cases

def _custom(lens, spec=wl.TINY, seed=0, **kw):
    return wl.generate(spec.replace(name="custom", batch=len(lens), lengths=("fixed", tuple(lens)),
                                    pool=("factor", 1.5), **kw), seed=seed)


@pytest.mark.parametrize("splits", [1, 2, 0])
def test_edge_lengths_block_and_split_boundaries(splits):
    # 1024-token table width: two splits put the boundary exactly at token 512.
    lens = (1, 15, 16, 17, 31, 32, 33, 511, 512, 513, 1024, 2)
    w = _custom(lens, spec=wl.LLAMA3_8B.replace(num_q_heads=8, num_kv_heads=2))
    assert w.max_blocks == 64
    full_check(w, splits)


@pytest.mark.parametrize("splits", [1, 3])
def test_empty_contexts_give_zero_rows(splits):
    w = _custom((0, 5, 0, 40))
    out, _, _ = run_gpu_step(w, 0, splits)
    o = out.float()
    assert torch.all(o[0] == 0) and torch.all(o[2] == 0)
    rk, rv = oracle_caches(w)
    ref = oracle_rows(w, rk, rv, [(1, 3), (3, 7)])
    assert_close(widen_out(out, "fp16")[[1, 3], [3, 7]], ref, "non-empty rows")


@pytest.mark.parametrize("splits", [1, 2])
def test_one_token_context_returns_v_bit_exact(splits):
    w = _custom((1, 1, 1), spec=wl.LLAMA3_8B.replace(num_q_heads=16, num_kv_heads=2))
    w.block_tables = np.concatenate([w.block_tables, np.full((3, 1), -1, np.int32)], axis=1)  # 2 columns
    out, _, vc = run_gpu_step(w, 0, splits)
    vnew = bits(w.v_new[0])
    o = bits(out)
    for b in range(3):
        for h in range(16):
            assert np.array_equal(o[b, h], vnew[b, h // 8])


def test_equal_keys_give_mean_of_v():
    w = _custom((100, 37))
    kc = w.k_cache[0]
    key = w.k_new[0][0, 0].clone()
    kc[:] = key                       # every cached key (and NaN slot) becomes the same key
    w.k_new[0][:] = key
    out, _, vc = run_gpu_step(w, 0, 1)
    rk, rv = oracle_caches(w)
    vmean = np.stack([oracle.widen(oracle.gather_kv(rv, w.block_tables[b], int(w.context_lens[b]), h // 4, 16),
                                   "fp16").mean(axis=0) for b in range(2) for h in range(8)]).reshape(2, 8, -1)
    assert_close(widen_out(out, "fp16"), vmean, "equal keys")


# ---------------------------------------------------------------- properties

def test_block_placement_permutation_gives_identical_bits():
    w = _custom((100, 7, 64, 33), spec=wl.LLAMA3_8B.replace(num_q_heads=16, num_kv_heads=4))
    a, _, _ = run_gpu_step(w, 0, 1)
    perm = np.random.default_rng(5).permutation(w.num_blocks)
    inv_perm = torch.from_numpy(np.argsort(perm))
    w.k_cache[0] = w.k_cache[0][inv_perm]  # block i moves to perm[i]
    w.v_cache[0] = w.v_cache[0][inv_perm]
    w.block_tables = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    b, _, _ = run_gpu_step(w, 0, 1)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_shared_prefix_blocks_equal_private_copies():
    spec = wl.LLAMA70B_TAIL.replace(name="share", batch=8, lengths=("uniform", 100, 300), shared_prefix=(4, 64))
    w = wl.generate(spec, seed=2)
    shared, _, _ = run_gpu_step(w, 0, 0)
    # give every sharing sequence private copies of the 4 prefix blocks
    kc, vc = w.k_cache[0], w.v_cache[0]
    free = sorted(set(range(w.num_blocks)) - set(int(x) for x in w.block_tables[w.block_tables >= 0]))
    tables = w.block_tables.copy()
    for b in w.shared_seqs[1:]:
        for j in range(4):
            dst = free.pop()
            kc[dst] = kc[tables[b, j]]
            vc[dst] = vc[tables[b, j]]
            tables[b, j] = dst
    w.block_tables = tables
    private, _, _ = run_gpu_step(w, 0, 0)
    assert torch.equal(shared.view(torch.int16), private.view(torch.int16))


def test_single_pass_and_splits_agree():
    w = wl.generate(wl.LLAMA3_8B.replace(batch=8), seed=4)
    rk, rv = oracle_caches(w)
    ref = oracle_rows(w, rk, rv, [(b, h) for b in range(8) for h in range(32)]).reshape(8, 32, -1)
    one = widen_out(run_gpu_step(w, 0, 1)[0], "bf16")
    assert_close(one, ref, "single pass")
    for n in (0, 2, 8, 256):
        many = widen_out(run_gpu_step(w, 0, n)[0], "bf16")
        assert_close(many, ref, f"{n} splits")
        # Each partition rounds its softmax weights to bf16 relative to its own
        # running max and rounds the output once more: two partitions differ
        # by a few bf16 steps of the output, far inside the oracle tolerance.
        diff = np.abs(one - many)
        bound = 2 ** -6 * np.maximum(np.abs(one), np.abs(many)) + 2 ** -11
        k = np.unravel_index(np.argmax(diff - bound), diff.shape)
        assert diff[k] <= bound[k], f"splits={n}: at {k} one={one[k]} many={many[k]} ref={ref[k]}"


def test_gqa_equals_mha_with_repeated_heads():
    w = _custom((70, 20, 129), spec=wl.LLAMA3_8B.replace(num_q_heads=8, num_kv_heads=2))
    gqa, _, _ = run_gpu_step(w, 0, 1)
    w.k_cache[0] = w.k_cache[0].repeat_interleave(4, dim=1).contiguous()
    w.v_cache[0] = w.v_cache[0].repeat_interleave(4, dim=1).contiguous()
    w.k_new[0] = w.k_new[0].repeat_interleave(4, dim=1).contiguous()
    w.v_new[0] = w.v_new[0].repeat_interleave(4, dim=1).contiguous()
    mha, _, _ = run_gpu_step(w, 0, 1)
    assert_close(widen_out(mha, "bf16"), widen_out(gqa, "bf16").astype(np.float64), "gqa vs mha")


# ---------------------------------------------------------------- host-produced tables and steps

def test_allocator_tables_end_to_end():
    """Block tables and slots from the C++ allocator, incl. a forked prefix."""
    spec = wl.LLAMA3_8B.replace(name="alloc", batch=6)
    D, Hk = spec.head_dim, spec.num_kv_heads
    alloc = pkv.BlockAllocator(200, 16, seed=9)
    lens_before = [300, 17, 0, 511, 600, 48]
    ids = [alloc.add_seq(L) for L in lens_before[:4]]
    ids.append(alloc.fork_prefix(ids[3], 496, 600))
    ids.append(alloc.fork_prefix(ids[1], 16, 48))
    slots = np.array([alloc.append_slot(s) for s in ids], np.int32)
    tables, lens = alloc.block_tables(ids, 40)
    g = torch.Generator().manual_seed(0)
    kc = torch.randn(200, Hk, 16, D, generator=g).to(torch.bfloat16)
    vc = torch.randn(200, Hk, 16, D, generator=g).to(torch.bfloat16)
    w = wl.Workload(spec=spec, seed=0, context_lens=lens, block_tables=tables, num_blocks=200,
                    scale=1 / math.sqrt(D), q=[torch.randn(6, 32, D, generator=g).to(torch.bfloat16)],
                    k_new=[torch.randn(6, Hk, D, generator=g).to(torch.bfloat16)],
                    v_new=[torch.randn(6, Hk, D, generator=g).to(torch.bfloat16)], k_cache=[kc], v_cache=[vc])
    assert np.array_equal(slots, oracle.slot_mapping(tables, lens, 16))
    out, kcg, vcg = run_gpu_step(w, 0, 0, slots=slots)
    rk, rv = oracle_caches(w)
    assert np.array_equal(bits(kcg), rk) and np.array_equal(bits(vcg), rv)
    rows = [(b, h) for b in range(6) for h in range(32)]
    assert_close(widen_out(out, "bf16").reshape(-1, D), oracle_rows(w, rk, rv, rows), "allocator tables")


def test_step_from_host_matches_device_calls():
    w = wl.generate(wl.LLAMA3_8B.replace(batch=5), seed=6)
    ref_out, ref_k, _ = run_gpu_step(w, 0, 0)
    dev = torch.device("cuda")
    kc = w.k_cache[0].to(dev, copy=True)
    vc = w.v_cache[0].to(dev, copy=True)
    host = {"q": w.q[0], "k_new": w.k_new[0], "v_new": w.v_new[0],
            "block_tables": torch.from_numpy(w.block_tables),
            "context_lens": torch.from_numpy(w.context_lens), "out": torch.empty_like(w.q[0])}
    host = {k: v.contiguous().pin_memory() for k, v in host.items()}
    devb = {k: torch.empty_like(v, device=dev) for k, v in host.items()}
    ws = pkv.make_workspace(devb["q"], kc, devb["block_tables"])
    pkv.paged_decode_step_from_host(host, devb, kc, vc, w.scale, 0, ws)
    torch.cuda.synchronize()
    assert torch.equal(host["out"].view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(kc.cpu().view(torch.int16), ref_k.view(torch.int16))


@pytest.mark.parametrize("layout", ["pinned", "packed", "pageable", "mixed"])
def test_step_from_host_chained_steps_match_device_calls(layout):
    """Several host-buffer steps issued back to back through the same device
    staging, each with its own host inputs and output buffer: every output
    and the final caches equal those of the same steps run from device
    tensors.  pinned: separate pinned buffers (kernel copies, 4-byte units for
    the 20-byte lengths); packed: one pinned buffer and one device region (a
    single merged copy); pageable: unpinned host memory (copy-engine copies);
    mixed: pinned inputs but pageable lengths and output (kernel copies, the
    decode kernel not launched early, a copy-engine copy of the output)."""
    w = wl.generate(wl.LLAMA3_8B.replace(batch=5), seed=6)
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(1)
    steps = []
    for _ in range(4):
        steps.append({"q": torch.randn(w.q[0].shape, generator=g).bfloat16(),
                      "k_new": torch.randn(w.k_new[0].shape, generator=g).bfloat16(),
                      "v_new": torch.randn(w.v_new[0].shape, generator=g).bfloat16(),
                      "block_tables": torch.from_numpy(w.block_tables).clone(),
                      "context_lens": torch.from_numpy(w.context_lens).clone()})
    kc_ref, vc_ref = w.k_cache[0].to(dev, copy=True), w.v_cache[0].to(dev, copy=True)
    ref_out = []
    for st in steps:
        d = {k: v.to(dev) for k, v in st.items()}
        ref_out.append(pkv.paged_decode_step(d["q"], d["k_new"], d["v_new"], kc_ref, vc_ref, d["block_tables"],
                                             d["context_lens"], w.scale).cpu())
    keys = ["q", "k_new", "v_new", "block_tables", "context_lens"]
    kc, vc = w.k_cache[0].to(dev, copy=True), w.v_cache[0].to(dev, copy=True)
    if layout == "packed":
        nbytes = [steps[0][k].numel() * steps[0][k].element_size() for k in keys]
        region = torch.empty(sum(nbytes), dtype=torch.uint8, device=dev)
        devb, off = {}, 0
        for k, n in zip(keys, nbytes):
            devb[k] = region[off:off + n].view(steps[0][k].dtype).view(steps[0][k].shape)
            off += n
    else:
        devb = {k: torch.empty_like(steps[0][k], device=dev) for k in keys}
    devb["out"] = torch.empty_like(steps[0]["q"], device=dev)
    hosts = []
    for st in steps:
        if layout == "packed":
            buf = torch.empty(sum(nbytes), dtype=torch.uint8).pin_memory()
            h, off = {}, 0
            for k, n in zip(keys, nbytes):
                h[k] = buf[off:off + n].view(st[k].dtype).view(st[k].shape)
                h[k].copy_(st[k])
                off += n
            h["_buf"] = buf
        else:
            pin = {"pinned": keys, "pageable": [], "mixed": ["q", "k_new", "v_new", "block_tables"]}[layout]
            h = {k: (st[k].contiguous().pin_memory() if k in pin else st[k].contiguous().clone()) for k in keys}
        h["out"] = torch.full_like(st["q"], float("nan"))
        if layout in ("pinned", "packed"):
            h["out"] = h["out"].pin_memory()
        hosts.append(h)
    ws = pkv.make_workspace(devb["q"], kc, devb["block_tables"])
    for h in hosts:
        pkv.paged_decode_step_from_host(h, devb, kc, vc, w.scale, 0, ws)
    torch.cuda.synchronize()
    pkv.paged_kv_check_status()
    for h, r in zip(hosts, ref_out):
        assert torch.equal(h["out"].view(torch.int16), r.view(torch.int16))
    assert torch.equal(kc.view(torch.int16), kc_ref.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), vc_ref.view(torch.int16))


# ---------------------------------------------------------------- errors

def test_out_of_range_inputs_are_flagged_not_faulted():
    w = _custom((40, 20))
    dev = torch.device("cuda")
    kc, vc = w.k_cache[0].to(dev), w.v_cache[0].to(dev)
    q = w.q[0].to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    slots = torch.from_numpy(pkv.paged_kv_slot_mapping(w.block_tables, w.context_lens)).to(dev)
    pkv.paged_kv_append(w.k_new[0].to(dev), w.v_new[0].to(dev), slots, kc, vc)  # fills slot L-1
    bad = w.block_tables.copy()
    bad[0, 1] = w.num_blocks + 5
    out = pkv.paged_decode_attention(q, kc, vc, torch.from_numpy(bad).to(dev), cl, w.scale, num_splits=1)
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_kv_check_status()
    assert e.value.code == -6
    assert torch.isfinite(out.float()).all()
    pkv.paged_kv_check_status()  # cleared
    # append slot past the pool: skipped and flagged
    slot = torch.tensor([w.num_blocks * 16, -1], dtype=torch.int32, device=dev)
    before = kc.clone()
    pkv.paged_kv_append(w.k_new[0].to(dev), w.v_new[0].to(dev), slot, kc, vc)
    with pytest.raises(pkv.PagedKVError):
        pkv.paged_kv_check_status()
    assert torch.equal(before.view(torch.int16), kc.view(torch.int16))
    # context longer than the table: clamped and flagged
    long = torch.tensor([10 ** 6, 20], dtype=torch.int32, device=dev)
    pkv.paged_decode_attention(q, kc, vc, torch.from_numpy(w.block_tables).to(dev), long, w.scale)
    with pytest.raises(pkv.PagedKVError):
        pkv.paged_kv_check_status()


def test_invalid_arguments_are_rejected():
    dev = torch.device("cuda")
    kc = torch.zeros(8, 2, 16, 96, dtype=torch.float16, device=dev)
    q = torch.zeros(1, 4, 96, dtype=torch.float16, device=dev)
    bt = torch.zeros(1, 2, dtype=torch.int32, device=dev)
    cl = torch.ones(1, dtype=torch.int32, device=dev)
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_decode_attention(q, kc, kc, bt, cl, 0.1)
    assert e.value.code == -2                     # head_dim 96 not compiled
    kc = torch.zeros(8, 1, 16, 64, dtype=torch.float16, device=dev)
    q = torch.zeros(1, 16, 64, dtype=torch.float16, device=dev)
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_decode_attention(q, kc, kc, bt, cl, 0.1)
    assert e.value.code == -2                     # 16 query heads per KV head
    q = torch.zeros(1, 3, 64, dtype=torch.float16, device=dev)
    kc2 = torch.zeros(8, 2, 16, 64, dtype=torch.float16, device=dev)
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_decode_attention(q, kc2, kc2, bt, cl, 0.1)
    assert e.value.code == -1                     # 2 does not divide 3
    q = torch.zeros(1, 4, 64, dtype=torch.float16, device=dev)
    small = torch.empty(4, dtype=torch.uint8, device=dev)
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_decode_attention(q, kc2, kc2, bt, cl, 0.1, num_splits=2, workspace=small)
    assert e.value.code == -1                     # workspace too small


# ---------------------------------------------------------------- persistent path

def test_persistent_path_is_selected_and_reuses_its_workspace():
    """num_splits=0 runs the balanced persistent kernel; its scheduler
    counters return to zero, so the same workspace serves call after call."""
    w = wl.generate(wl.LLAMA3_8B.replace(batch=24), seed=8)
    dev = torch.device("cuda")
    kc, vc = w.k_cache[0].to(dev), w.v_cache[0].to(dev)
    q = w.q[0].to(dev)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    assert pkv.paged_decode_resolve_splits(q, kc, bt, 0) == 0
    slots = torch.from_numpy(pkv.paged_kv_slot_mapping(w.block_tables, w.context_lens)).to(dev)
    pkv.paged_kv_append(w.k_new[0].to(dev), w.v_new[0].to(dev), slots, kc, vc)
    ws = pkv.make_workspace(q, kc, bt, 0)
    outs = [pkv.paged_decode_attention(q, kc, vc, bt, cl, w.scale, num_splits=0, workspace=ws) for _ in range(3)]
    pkv.paged_kv_check_status()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    sched = ws[-256:].view(torch.int32)   # scheduler counters: the last region
    assert int(sched.abs().sum()) == 0
    rk, rv = oracle_caches(w)
    rows = sample_rows(w, 40)
    gpu = widen_out(outs[0].cpu(), "bf16")
    assert_close(np.stack([gpu[b, h] for b, h in rows]), oracle_rows(w, rk, rv, rows), "persistent")


def test_large_batch_falls_back_to_splits():
    """More sequences than the persistent kernel's shared-memory plan holds:
    the automatic path uses 512-token splits and stays exact."""
    spec = wl.TINY.replace(name="wide", batch=2100, lengths=("uniform", 1, 40), pool=("factor", 1.2))
    w = wl.generate(spec, seed=1)
    dev = torch.device("cuda")
    assert pkv.paged_decode_resolve_splits(w.q[0].to(dev), w.k_cache[0].to(dev),
                                           torch.from_numpy(w.block_tables).to(dev), 0) >= 1
    full_check(w, 0, rows=sample_rows(w, 64))


@pytest.mark.parametrize("head_dim", [128, 64])
def test_persistent_path_at_its_largest_batch(head_dim):
    """2048 sequences, the most the persistent kernel's shared-memory plan
    holds: still the persistent path, every output and the append exact, for
    the fused step and for append + attention."""
    spec = wl.LLAMA3_8B.replace(name="b2048", batch=2048, lengths=("uniform", 1, 40), num_q_heads=8,
                                num_kv_heads=2, head_dim=head_dim, pool=("factor", 1.2))
    w = wl.generate(spec, seed=6)
    dev = torch.device("cuda")
    assert pkv.paged_decode_resolve_splits(w.q[0].to(dev), w.k_cache[0].to(dev),
                                           torch.from_numpy(w.block_tables).to(dev), 0) == 0
    full_check_every_output(w, 0)
    full_check(w, 0, fused=True, rows=sample_rows(w, 256))


@pytest.mark.parametrize("lens", [(1,), (5, 0, 7), (16,) * 3, (4096, 1, 1, 1), (0, 0)])
def test_persistent_short_and_uneven_batches(lens):
    w = _custom(lens, spec=wl.LLAMA3_8B.replace(num_q_heads=8, num_kv_heads=2))
    if max(lens) == 0:
        out, _, _ = run_gpu_step(w, 0, 0)
        assert torch.all(out.float() == 0)
        return
    full_check(w, 0)


# ---------------------------------------------------------------- fused decode step

@pytest.mark.parametrize("splits", [0, 5])
@pytest.mark.parametrize("spec", [wl.TINY] + REDUCED, ids=lambda s: s.name)
def test_fused_step_every_output(spec, splits):
    """paged_decode_step (append at position L-1 + attention, one call) gives
    the oracle's append bit for bit and its attention within tolerance."""
    w = wl.generate(spec, seed=5)
    for layer in range(len(w.q)):
        full_check(w, splits, layer, fused=True)


def test_fused_step_llama3_8b_full_every_output():
    full_check(wl.generate(wl.LLAMA3_8B, seed=2, device="cuda"), 0, fused=True)


@pytest.mark.parametrize("spec", [wl.LLAMA70B_TAIL, wl.LONG_CTX, wl.MHA_7B_B64], ids=lambda s: s.name)
def test_fused_step_full_sampled(spec):
    w = wl.generate(spec, seed=3, device="cuda", layers=1)
    rows = sample_rows(w, 64) + [(b, 0) for b in range(min(8, w.spec.batch))]
    full_check(w, 0, rows=sorted(set(rows)), fused=True)


@pytest.mark.parametrize("lens", [(1,), (5, 0, 7), (16,) * 3, (17, 1, 33), (4096, 1, 1, 1)])
def test_fused_step_edge_lengths(lens):
    w = _custom(lens, spec=wl.LLAMA3_8B.replace(num_q_heads=8, num_kv_heads=2))
    full_check(w, 0, fused=True)


def test_fused_and_separate_steps_give_identical_bits():
    w = wl.generate(wl.LLAMA3_8B.replace(batch=12), seed=9)
    a, ka, va = run_gpu_step(w, 0, 0, fused=False)
    b, kb, vb = run_gpu_step(w, 0, 0, fused=True)
    assert torch.equal(ka.view(torch.int16), kb.view(torch.int16))
    assert torch.equal(va.view(torch.int16), vb.view(torch.int16))
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_bounded_wait_gives_up_reports_timeout_and_the_device_stays_usable():
    """A wait on a barrier nothing signals: the kernel gives up after its limit,
    the host reads PKV_ERR_TIMEOUT, and the next decode is still correct."""
    import time
    t0 = time.time()
    pkv.paged_kv_selftest_wait()
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_kv_check_status()
    assert e.value.code == -4 and "bounded wait" in str(e.value)
    assert 1.0 < time.time() - t0 < 30.0
    pkv.paged_kv_check_status()  # cleared
    full_check(wl.generate(wl.TINY, seed=4), 0)


@pytest.mark.parametrize("fp8", [False, True])
def test_decode_step_replays_from_a_cuda_graph(fp8):
    """A step captured in a CUDA graph and replayed gives the same bits as the
    direct call (the step is idempotent: same token, same slot)."""
    spec = wl.LLAMA3_8B.replace(name="graph", batch=9, lengths=("uniform", 1, 600), num_q_heads=16,
                                num_kv_heads=4)
    w = wl.generate(spec, seed=6)
    dev = torch.device("cuda")
    q, kn, vn = w.q[0].to(dev), w.k_new[0].to(dev), w.v_new[0].to(dev)
    bt, cl = torch.from_numpy(w.block_tables).to(dev), torch.from_numpy(w.context_lens).to(dev)
    if fp8:
        f8 = wl.fp8_caches(w, seed=6)
        kc, vc = f8.k_cache[0].to(dev, copy=True), f8.v_cache[0].to(dev, copy=True)
        ks, vs = f8.k_scale[0].to(dev), f8.v_scale[0].to(dev)
        ws = torch.zeros(pkv.paged_decode_workspace_bytes(q, w.k_cache[0], bt, 0), dtype=torch.uint8, device=dev)

        def step(out, stream=None):
            pkv.paged_decode_step_fp8(q, kn, vn, kc, vc, ks, vs, bt, cl, w.scale, out=out, workspace=ws,
                                      stream=stream)
    else:
        kc, vc = w.k_cache[0].to(dev, copy=True), w.v_cache[0].to(dev, copy=True)
        ws = pkv.make_workspace(q, kc, bt, 0)

        def step(out, stream=None):
            pkv.paged_decode_step(q, kn, vn, kc, vc, bt, cl, w.scale, out=out, workspace=ws, stream=stream)

    direct = torch.empty_like(q)
    step(direct)
    torch.cuda.synchronize()
    replayed = torch.zeros_like(q)
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=cap):
        step(replayed, stream=cap)
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    pkv.paged_kv_check_status()
    assert torch.equal(direct.view(torch.int16), replayed.view(torch.int16))

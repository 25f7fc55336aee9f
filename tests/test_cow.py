"""Copy-on-write of shared blocks: the allocator's forks and copy decisions
(host, no GPU), and, on the GPU, the block-copy kernel and a parallel-sampling
decode loop checked against the oracle.

The page's rule (kasblo.com "vLLMとは？", section "block共有とAutomatic Prefix
Caching"): a block carries a reference count, several sequences may hold it,
and it is duplicated only when one of them must write into it."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_26_gb300 as pkv
from paged_kv_cache_26_gb300 import BlockAllocator, PagedKVError
from paged_kv_cache_26_gb300 import build as pkv_build

BS = 16


@pytest.fixture(scope="module", autouse=True)
def built():
    pkv_build.build()


def tables_of(a, ids, mb):
    return a.block_tables(ids, mb)


# ---------------------------------------------------------------- allocator (host)

def test_fork_shares_blocks_and_writes_copy_once():
    a = BlockAllocator(20, BS, seed=1)
    src = a.add_seq(37)                                   # blocks: 2 full + 1 holding 5 tokens
    t_src, _ = tables_of(a, [src], 3)
    free0 = a.num_free
    f = a.fork(src, 37)
    t_f, l_f = tables_of(a, [f], 3)
    assert list(t_f[0]) == list(t_src[0]) and l_f[0] == 37 and a.num_free == free0
    assert all(a.refcount(int(b)) == 2 for b in t_src[0])
    slot, copy = a.append_slot_cow(f)                     # position 37 lands in the shared third block
    old = int(t_src[0][2])
    assert copy is not None and copy[0] == old
    fresh = copy[1]
    assert slot == fresh * BS + 37 % BS and a.refcount(old) == 1 and a.refcount(fresh) == 1
    assert list(tables_of(a, [f], 3)[0][0]) == [int(t_src[0][0]), int(t_src[0][1]), fresh]
    assert a.append_slot_cow(f)[1] is None                # now private
    slot_s, copy_s = a.append_slot_cow(src)               # the source keeps the original in place
    assert copy_s is None and slot_s == old * BS + 37 % BS
    assert a.refcount(int(t_src[0][0])) == 2              # full blocks stay shared


def test_fork_at_a_block_boundary_needs_no_copy_and_strict_append_refuses_shared():
    a = BlockAllocator(20, BS, seed=2)
    src = a.add_seq(40)
    f = a.fork(src, 32)
    assert a.seq_len(f) == 32
    slot, copy = a.append_slot_cow(f)
    assert copy is None and a.seq_len(f) == 33
    g = a.fork(src, 40)
    with pytest.raises(PagedKVError) as e:
        a.append_slot(g)                                  # the copy-free call refuses a shared block
    assert e.value.code == -7
    with pytest.raises(PagedKVError):
        a.fork(src, 41)                                   # longer than the source


def test_step_batch_cow_parallel_sampling_copies_all_but_one():
    a = BlockAllocator(30, BS, seed=3)
    src = a.add_seq(21)
    forks = [a.fork(src, 21) for _ in range(4)]
    shared = int(tables_of(a, [src], 2)[0][0][1])
    assert a.refcount(shared) == 5
    ids = np.array([src] + forks, np.int32)
    tables = np.empty((5, 4), np.int32)
    lens = np.empty(5, np.int32)
    pairs = np.empty((5, 2), np.int32)
    free0 = a.num_free
    n = a.step_batch_cow(ids, 4, tables, lens, pairs)
    assert n == 4 and a.num_free == free0 - 4
    assert set(pairs[:n, 0]) == {shared} and len(set(pairs[:n, 1])) == 4
    assert sorted(tables[:, 1]) == sorted([shared] + list(pairs[:n, 1]))   # one holder kept the original
    assert all(a.refcount(int(b)) == 1 for b in tables[:, 1]) and np.all(lens == 22)
    assert a.refcount(int(tables[0, 0])) == 5                               # the full first block stays shared
    assert a.step_batch_cow(ids, 4, tables, lens, pairs) == 0               # every writer now private


def test_step_batch_cow_is_all_or_nothing():
    a = BlockAllocator(4, BS, seed=4)
    src = a.add_seq(20)                                   # 2 blocks
    forks = [a.fork(src, 20) for _ in range(3)]           # 3 copies needed, 2 free
    ids = np.array([src] + forks, np.int32)
    before = [list(tables_of(a, [s], 2)[0][0]) for s in ids]
    with pytest.raises(PagedKVError) as e:
        a.step_batch_cow(ids, 2, np.empty((4, 2), np.int32), np.empty(4, np.int32), np.empty((4, 2), np.int32))
    assert e.value.code == -5
    assert [list(tables_of(a, [s], 2)[0][0]) for s in ids] == before and a.num_free == 2
    assert [a.seq_len(int(s)) for s in ids] == [20] * 4


def test_parallel_sampling_simulation_keeps_every_sequence_intact():
    """The allocator drives 30 copy-on-write steps of a prompt, three samples
    forked from it and a shorter reuse; the oracle performs each step's copies
    and appends on a host pool.  Every sequence then reads its prefix plus its
    own tokens, and the reference counts match the tables."""
    rng = np.random.default_rng(9)
    D, Hkv, nb, mb = 8, 2, 40, 8
    a = BlockAllocator(nb, BS, seed=5)
    src = a.add_seq(0)
    prompt = rng.integers(0, 0x3C00, size=(27, Hkv, D), dtype=np.uint16)
    kc = np.full((nb, Hkv, BS, D), 0x7E00, np.uint16)
    vc = kc.copy()
    slots = [a.append_slot(src) for _ in range(27)]       # written while src is the only holder
    kc, vc = oracle.kv_append(kc, vc, prompt, prompt ^ 1, np.array(slots), BS)
    ids = np.array([src] + [a.fork(src, 27) for _ in range(3)] + [a.fork(src, 20)], np.int32)
    tables = np.empty((5, mb), np.int32)
    lens = np.empty(5, np.int32)
    pairs = np.empty((5, 2), np.int32)
    own = [[] for _ in range(5)]
    for _ in range(30):
        n = a.step_batch_cow(ids, mb, tables, lens, pairs)
        kc, vc = oracle.copy_blocks(kc, vc, [tuple(p) for p in pairs[:n]])
        k_new = rng.integers(0, 0x3C00, size=(5, Hkv, D), dtype=np.uint16)
        kc, vc = oracle.kv_append(kc, vc, k_new, k_new ^ 1, oracle.slot_mapping(tables, lens, BS), BS)
        for i in range(5):
            own[i].append(k_new[i])
    for i in range(5):
        expect = np.concatenate([prompt[:20 if i == 4 else 27], np.stack(own[i])])
        for kv in range(Hkv):
            assert np.array_equal(oracle.gather_kv(kc, tables[i], int(lens[i]), kv, BS), expect[:, kv])
            assert np.array_equal(oracle.gather_kv(vc, tables[i], int(lens[i]), kv, BS), expect[:, kv] ^ 1)
    held = {}
    for i in range(5):
        for blk in tables[i, :math.ceil(lens[i] / BS)]:
            held[int(blk)] = held.get(int(blk), 0) + 1
    assert all(a.refcount(blk) == c for blk, c in held.items())
    assert a.num_free + len(held) == nb


# ---------------------------------------------------------------- GPU

@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["bf16_d128", "fp16_d64", "e4m3_d128"])
def test_copy_blocks_kernel_bit_exact(kind):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(1)
    nb, hkv = 300, 8
    d = 64 if kind == "fp16_d64" else 128
    if kind == "e4m3_d128":
        kc = torch.randint(0, 256, (nb, hkv, BS, d), generator=g, dtype=torch.uint8)
        vc = torch.randint(0, 256, (nb, hkv, BS, d), generator=g, dtype=torch.uint8)
    else:
        dt = torch.bfloat16 if kind == "bf16_d128" else torch.float16
        kc = torch.randn(nb, hkv, BS, d, generator=g).to(dt)
        vc = torch.randn(nb, hkv, BS, d, generator=g).to(dt)
    perm = np.random.default_rng(2).permutation(nb)
    pairs = np.stack([perm[:120], perm[120:240]], 1).astype(np.int32)     # distinct dsts, none a source
    kd, vd = kc.to(dev), vc.to(dev)
    pkv.paged_kv_copy_blocks(kd, vd, torch.from_numpy(pairs).to(dev))
    pkv.paged_kv_check_status()
    view = (lambda t: t.view(torch.int16).numpy()) if kc.dtype != torch.uint8 else (lambda t: t.numpy())
    rk, rv = oracle.copy_blocks(view(kc), view(vc), [tuple(p) for p in pairs])
    assert np.array_equal(view(kd.cpu()), rk) and np.array_equal(view(vd.cpu()), rv)
    # a pair outside the pool is skipped and flagged
    before = kd.clone()
    pkv.paged_kv_copy_blocks(kd, vd, torch.tensor([[0, nb], [-1, 3]], dtype=torch.int32, device=dev))
    with pytest.raises(PagedKVError) as e:
        pkv.paged_kv_check_status()
    assert e.value.code == -6 and torch.equal(before, kd)


@pytest.mark.gpu
def test_parallel_sampling_decode_loop_against_the_oracle():
    """A prompt, four samples forked from it and one shorter reuse, decoded for
    40 steps with copy-on-write: every sequence's K/V is its prefix plus its own
    tokens, and the last step's attention matches the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda")
    Hq, Hkv, D, nb, mb = 8, 2, 128, 64, 8
    g = torch.Generator().manual_seed(3)
    dt = torch.bfloat16
    kc = torch.full((nb, Hkv, BS, D), float("nan"), dtype=dt, device=dev)
    vc = kc.clone()
    a = BlockAllocator(nb, BS, seed=7)
    src = a.add_seq(0)
    P = 45
    pk = torch.randn(P, Hkv, D, generator=g).to(dt)
    pv = torch.randn(P, Hkv, D, generator=g).to(dt)
    slots = torch.tensor([a.append_slot(src) for _ in range(P)], dtype=torch.int32, device=dev)
    pkv.paged_kv_append(pk.to(dev), pv.to(dev), slots, kc, vc)
    ids = np.array([src] + [a.fork(src, P) for _ in range(4)] + [a.fork(src, 33)], np.int32)
    B = len(ids)
    tables = np.empty((B, mb), np.int32)
    lens = np.empty(B, np.int32)
    pairs = np.empty((B, 2), np.int32)
    hist = {i: ([pk[t] for t in range(P if i < 5 else 33)], [pv[t] for t in range(P if i < 5 else 33)])
            for i in range(B)}
    total_copies = 0
    for step in range(40):
        n = a.step_batch_cow(ids, mb, tables, lens, pairs)
        total_copies += n
        if n:
            pkv.paged_kv_copy_blocks(kc, vc, torch.from_numpy(pairs[:n].copy()).to(dev))
        q = torch.randn(B, Hq, D, generator=g).to(dt)
        kn = torch.randn(B, Hkv, D, generator=g).to(dt)
        vn = torch.randn(B, Hkv, D, generator=g).to(dt)
        out = pkv.paged_decode_step(q.to(dev), kn.to(dev), vn.to(dev), kc, vc, torch.from_numpy(tables).to(dev),
                                    torch.from_numpy(lens).to(dev), 1 / math.sqrt(D))
        for i in range(B):
            hist[i][0].append(kn[i])
            hist[i][1].append(vn[i])
    pkv.paged_kv_check_status()
    assert total_copies >= 5                              # the shared partial blocks were copied

    def b16(t):
        return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)

    kcb, vcb = b16(kc), b16(vc)
    got = oracle.widen(b16(out), "bf16")
    for i in range(B):
        L = int(lens[i])
        K = b16(torch.stack(hist[i][0]))
        V = b16(torch.stack(hist[i][1]))
        assert L == K.shape[0]
        for kv in range(Hkv):
            assert np.array_equal(oracle.gather_kv(kcb, tables[i], L, kv, BS), K[:, kv])
            assert np.array_equal(oracle.gather_kv(vcb, tables[i], L, kv, BS), V[:, kv])
            for h in range(kv * Hq // Hkv, (kv + 1) * Hq // Hkv):
                ref = oracle.attend_one(oracle.widen(b16(q[i, h]), "bf16"), oracle.widen(K[:, kv], "bf16"),
                                        oracle.widen(V[:, kv], "bf16"), 1 / math.sqrt(D))[0]
                assert np.all(np.abs(got[i, h] - ref) <= 2e-3 + 1e-2 * np.abs(ref))

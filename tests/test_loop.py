"""Continuous batching: the allocator's batched growth (CPU) and a multi-step
decode loop checked end to end against the oracle (GPU).

The GPU test keeps, on the host, every token each sequence received (its
prompt plus one token per step).  After many steps with admissions,
retirements and block reuse, every live sequence's K/V read back through its
block table must equal that record bit for bit, and the last step's output
must match the oracle's attention over the record."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_26_gb300 import BlockAllocator, PagedKVError
from paged_kv_cache_26_gb300 import build as pkv_build


@pytest.fixture(scope="module", autouse=True)
def built():
    pkv_build.build()


def test_append_slots_batch_equals_single_appends():
    a1, a2 = BlockAllocator(50, 16, seed=4), BlockAllocator(50, 16, seed=4)
    ids1 = [a1.add_seq(n) for n in (0, 15, 16, 31, 40)]
    ids2 = [a2.add_seq(n) for n in (0, 15, 16, 31, 40)]
    for _ in range(40):
        batch = a1.append_slots(ids1)
        single = [a2.append_slot(s) for s in ids2]
        assert list(batch) == single
    assert a1.num_free == a2.num_free


def test_append_slots_is_all_or_nothing():
    a = BlockAllocator(4, 16, seed=0)
    ids = [a.add_seq(16), a.add_seq(16), a.add_seq(16)]     # 3 of 4 blocks used, all full
    before = [a.seq_len(s) for s in ids]
    with pytest.raises(PagedKVError) as e:
        a.append_slots(ids)                                 # needs 3 new blocks, 1 free
    assert e.value.code == -5
    assert [a.seq_len(s) for s in ids] == before and a.num_free == 1
    with pytest.raises(PagedKVError):
        a.append_slots([ids[0], ids[0]])                    # listed twice
    assert a.seq_len(ids[0]) == 16
    a.free_seq(ids[2])
    a.append_slots(ids[:2])
    assert [a.seq_len(s) for s in ids[:2]] == [17, 17]


def test_step_batch_grows_and_exports_every_slot():
    a, b = BlockAllocator(60, 16, seed=8), BlockAllocator(60, 16, seed=8)
    lens0 = (5, 16, 0, 47)
    ida = [a.add_seq(n) for n in lens0]
    idb = [b.add_seq(n) for n in lens0]
    slot_ids = np.array([ida[0], -1, ida[1], ida[2], -1, ida[3]], np.int32)
    tables = np.empty((6, 8), np.int32)
    lens = np.empty(6, np.int32)
    for _ in range(20):
        a.step_batch(slot_ids, 8, tables, lens)
        b.append_slots(idb)
        t_ref, l_ref = b.block_tables(idb, 8)
        live = [0, 2, 3, 5]
        assert np.array_equal(tables[live], t_ref) and np.array_equal(lens[live], l_ref)
        assert np.all(tables[[1, 4]] == -1) and np.all(lens[[1, 4]] == 0)
    with pytest.raises(PagedKVError):
        a.step_batch(slot_ids, 4, np.empty((6, 4), np.int32), lens)   # 47+20 tokens > 4 blocks
    assert a.seq_len(ida[3]) == 67


@pytest.mark.gpu
def test_decode_loop_end_to_end_against_the_oracle():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_26_gb300.loop import DecodeLoop

    dev = torch.device("cuda")
    Hq, Hk, D, B = 8, 2, 64, 6
    rng = np.random.default_rng(0)
    g = torch.Generator(device=dev).manual_seed(0)
    loop = DecodeLoop(num_blocks=40, num_q_heads=Hq, num_kv_heads=Hk, head_dim=D, max_batch=B,
                      max_context=200, dtype=torch.float16, device=dev, seed=3)
    history = {}                                            # sequence id -> list of (k, v) rows [Hk][D]

    def bits(t):
        return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)

    admitted = retired = 0
    q = None
    expect = {"steps": 0, "sequence_steps": 0, "context_tokens": 0, "unused_tail_slots": 0, "copied_blocks": 0}
    for step in range(70):
        # admit while there is room (prompts of 0..45 tokens, 3..30 steps each)
        assert loop.num_free_slots == loop.free_slots().size
        while loop.free_slots().size:
            P = int(rng.integers(0, 46))
            pk = torch.randn(P, Hk, D, generator=g, device=dev).half()
            pv = torch.randn(P, Hk, D, generator=g, device=dev).half()
            slot = loop.admit(pk, pv, int(rng.integers(3, 31)))
            if slot is None:
                break
            sid = int(loop.seq[slot])
            history[sid] = [(r[0], r[1]) for r in zip(bits(pk), bits(pv))]
            admitted += 1
        q = torch.randn(B, Hq, D, generator=g, device=dev).half()
        kn = torch.randn(B, Hk, D, generator=g, device=dev).half()
        vn = torch.randn(B, Hk, D, generator=g, device=dev).half()
        out = loop.step(q, kn, vn)
        for slot in loop.active_slots():
            history[int(loop.seq[slot])].append((bits(kn[slot]), bits(vn[slot])))
        Ls = loop.context_lengths()
        assert np.array_equal(loop.last_step()[1], Ls)
        act = Ls[Ls > 0]
        expect["steps"] += 1
        expect["sequence_steps"] += act.size
        expect["context_tokens"] += int(act.sum())
        expect["unused_tail_slots"] += int((-(-act // 16) * 16 - act).sum())
        if step < 69:
            retired += len(loop.finish_step())
    torch.cuda.synchronize()
    assert loop.stats() == expect
    loop.reset_stats()
    assert loop.stats() == dict.fromkeys(expect, 0)
    assert admitted > 2 * B and retired > B                  # sequences came and went, blocks were reused
    assert loop.waste_blocks() < 1.0

    kc, vc = bits(loop.k_cache), bits(loop.v_cache)
    tables, lens = loop.last_step()
    ref = np.zeros((B, Hq, D))
    got = oracle.widen(bits(out), "fp16")
    for slot in range(B):
        sid = int(loop.seq[slot])
        if sid < 0:
            assert lens[slot] == 0 and np.all(got[slot] == 0)
            continue
        hist = history[sid]
        L = len(hist)
        assert lens[slot] == L
        for kv in range(Hk):
            k_rec = np.stack([h[0][kv] for h in hist])
            v_rec = np.stack([h[1][kv] for h in hist])
            assert np.array_equal(oracle.gather_kv(kc, tables[slot], L, kv, 16), k_rec)
            assert np.array_equal(oracle.gather_kv(vc, tables[slot], L, kv, 16), v_rec)
            for h in range(kv * (Hq // Hk), (kv + 1) * (Hq // Hk)):
                ref[slot, h] = oracle.attend_one(oracle.widen(bits(q[slot, h]), "fp16"), oracle.widen(k_rec, "fp16"),
                                                 oracle.widen(v_rec, "fp16"), 1 / math.sqrt(D))[0]
    assert np.all(np.abs(got - ref) <= 2e-3 + 1e-2 * np.abs(ref))
    # every block is either free or held by exactly the live sequences' tables
    live_blocks = set(int(x) for s in range(B) if loop.seq[s] >= 0 for x in tables[s, :math.ceil(lens[s] / 16)])
    assert loop.alloc.num_free + len(live_blocks) == 40


@pytest.mark.gpu
def test_decode_loop_with_parallel_sampling_against_the_oracle():
    """Forks (parallel samples) of live sequences share their blocks; the loop
    copies a shared block before a step writes into it.  Every sequence must
    read back exactly its own history and the output match the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_26_gb300.loop import DecodeLoop

    dev = torch.device("cuda")
    Hq, Hk, D, B = 8, 2, 128, 8
    rng = np.random.default_rng(1)
    g = torch.Generator(device=dev).manual_seed(1)
    loop = DecodeLoop(num_blocks=80, num_q_heads=Hq, num_kv_heads=Hk, head_dim=D, max_batch=B,
                      max_context=160, dtype=torch.bfloat16, device=dev, seed=5)
    history = {}

    def bits(t):
        return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)

    forks = 0
    q = out = None
    for step in range(50):
        while loop.free_slots().size:
            active = loop.active_slots()
            if active.size and rng.random() < 0.6:
                src = int(rng.choice(active))
                slot = loop.fork(src, int(rng.integers(3, 25)))
                if slot is None:
                    break
                history[int(loop.seq[slot])] = list(history[int(loop.seq[src])])
                forks += 1
            else:
                P = int(rng.integers(1, 40))
                pk = torch.randn(P, Hk, D, generator=g, device=dev).bfloat16()
                pv = torch.randn(P, Hk, D, generator=g, device=dev).bfloat16()
                slot = loop.admit(pk, pv, int(rng.integers(3, 25)))
                if slot is None:
                    break
                history[int(loop.seq[slot])] = [(r[0], r[1]) for r in zip(bits(pk), bits(pv))]
        q = torch.randn(B, Hq, D, generator=g, device=dev).bfloat16()
        kn = torch.randn(B, Hk, D, generator=g, device=dev).bfloat16()
        vn = torch.randn(B, Hk, D, generator=g, device=dev).bfloat16()
        out = loop.step(q, kn, vn)
        for slot in loop.active_slots():
            history[int(loop.seq[slot])].append((bits(kn[slot]), bits(vn[slot])))
        if step < 49:
            loop.finish_step()
    torch.cuda.synchronize()
    assert forks > B
    assert loop.stats()["copied_blocks"] > 0                # shared blocks were copied before writes
    kc, vc = bits(loop.k_cache), bits(loop.v_cache)
    tables, lens = loop.last_step()
    got = oracle.widen(bits(out), "bf16")
    for slot in range(B):
        sid = int(loop.seq[slot])
        if sid < 0:
            continue
        hist = history[sid]
        L = len(hist)
        assert lens[slot] == L
        for kv in range(Hk):
            k_rec = np.stack([h[0][kv] for h in hist])
            v_rec = np.stack([h[1][kv] for h in hist])
            assert np.array_equal(oracle.gather_kv(kc, tables[slot], L, kv, 16), k_rec)
            assert np.array_equal(oracle.gather_kv(vc, tables[slot], L, kv, 16), v_rec)
            for h in range(kv * (Hq // Hk), (kv + 1) * (Hq // Hk)):
                ref = oracle.attend_one(oracle.widen(bits(q[slot, h]), "bf16"), oracle.widen(k_rec, "bf16"),
                                        oracle.widen(v_rec, "bf16"), 1 / math.sqrt(D))[0]
                assert np.all(np.abs(got[slot, h] - ref) <= 2e-3 + 1e-2 * np.abs(ref))


@pytest.mark.gpu
def test_decode_loop_on_an_fp8_pool_with_forks_against_the_oracle():
    """The loop over an E4M3 pool: every sequence's codes are the oracle's
    quantisation of its history (forks included), and the output matches the
    oracle's attention over the dequantised pool."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_26_gb300.loop import DecodeLoop

    dev = torch.device("cuda")
    Hq, Hk, D, B = 8, 2, 128, 6
    rng = np.random.default_rng(2)
    g = torch.Generator(device=dev).manual_seed(2)
    ks = torch.tensor([0.011, 0.017], dtype=torch.float32, device=dev)
    vs = torch.tensor([0.013, 0.009], dtype=torch.float32, device=dev)
    loop = DecodeLoop(num_blocks=60, num_q_heads=Hq, num_kv_heads=Hk, head_dim=D, max_batch=B, max_context=128,
                      dtype=torch.bfloat16, device=dev, seed=9, k_scale=ks, v_scale=vs)
    history = {}

    def bits(t):
        return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)

    forks = 0
    q = out = None
    for step in range(30):
        while loop.free_slots().size:
            active = loop.active_slots()
            if active.size and rng.random() < 0.5:
                src = int(rng.choice(active))
                slot = loop.fork(src, int(rng.integers(3, 20)))
                if slot is None:
                    break
                history[int(loop.seq[slot])] = list(history[int(loop.seq[src])])
                forks += 1
            else:
                P = int(rng.integers(1, 40))
                pk = torch.randn(P, Hk, D, generator=g, device=dev).bfloat16()
                pv = torch.randn(P, Hk, D, generator=g, device=dev).bfloat16()
                slot = loop.admit(pk, pv, int(rng.integers(3, 20)))
                if slot is None:
                    break
                history[int(loop.seq[slot])] = [(r[0], r[1]) for r in zip(bits(pk), bits(pv))]
        q = torch.randn(B, Hq, D, generator=g, device=dev).bfloat16()
        kn = torch.randn(B, Hk, D, generator=g, device=dev).bfloat16()
        vn = torch.randn(B, Hk, D, generator=g, device=dev).bfloat16()
        out = loop.step(q, kn, vn)
        for slot in loop.active_slots():
            history[int(loop.seq[slot])].append((bits(kn[slot]), bits(vn[slot])))
        if step < 29:
            loop.finish_step()
    torch.cuda.synchronize()
    assert forks > 0
    kc, vc = loop.k_cache.cpu().numpy(), loop.v_cache.cpu().numpy()
    tables, lens = loop.last_step()
    ksn, vsn = ks.cpu().numpy(), vs.cpu().numpy()
    got = oracle.widen(bits(out), "bf16")
    for slot in range(B):
        sid = int(loop.seq[slot])
        if sid < 0:
            continue
        hist = history[sid]
        L = len(hist)
        assert lens[slot] == L
        for kv in range(Hk):
            k_codes = oracle.quantize_e4m3(np.stack([h[0][kv] for h in hist]), "bf16", ksn[kv])
            v_codes = oracle.quantize_e4m3(np.stack([h[1][kv] for h in hist]), "bf16", vsn[kv])
            assert np.array_equal(oracle.gather_kv(kc, tables[slot], L, kv, 16), k_codes)
            assert np.array_equal(oracle.gather_kv(vc, tables[slot], L, kv, 16), v_codes)
            K = oracle.dequantize_e4m3(k_codes, ksn[kv])
            V = oracle.dequantize_e4m3(v_codes, vsn[kv])
            for h in range(kv * (Hq // Hk), (kv + 1) * (Hq // Hk)):
                ref = oracle.attend_one(oracle.widen(bits(q[slot, h]), "bf16"), K, V, 1 / math.sqrt(D))[0]
                assert np.all(np.abs(got[slot, h] - ref) <= 2e-3 + 1e-2 * np.abs(ref))

"""Host-side checks that need no GPU: the library builds for sm_103a, loads,
exports every function include/paged_kv.h declares; the block allocator and
the host slot mapping behave as the pages describe (compared with the oracle
and the pages' block-table example)."""
import ctypes
import json
import os
import re

import numpy as np
import pytest

import oracle
import paged_kv_cache_26_gb300 as pkv
from paged_kv_cache_26_gb300 import BlockAllocator, PagedKVError, paged_kv_slot_mapping
from paged_kv_cache_26_gb300 import build as pkv_build
from paged_kv_cache_26_gb300._native import EXPORTED

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    pkv_build.build()


def header_functions():
    text = open(os.path.join(ROOT, "include", "paged_kv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)) - {"if", "sizeof"})


def test_library_exports_every_declared_function():
    lib = ctypes.CDLL(pkv_build.LIB_PATH)
    declared = header_functions()
    assert len(declared) >= 17
    for name in declared:
        assert hasattr(lib, name), name
    assert set(declared) == set(EXPORTED)


def test_library_is_built_for_sm_103a_only():
    # Every translation unit is compiled with this one -gencode and no other.
    assert pkv_build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert "-lineinfo" in pkv_build.COMMON


def header_prototypes():
    """Parameter count of every function the header declares."""
    text = open(os.path.join(ROOT, "include", "paged_kv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"#.*", "", text)
    protos = {}
    for m in re.finditer(r"\b([a-z_][a-z0-9_]*)\s*\(([^;{}]*?)\)\s*;", text):
        name, params = m.group(1), m.group(2).strip()
        protos[name] = 0 if params in ("", "void") else params.count(",") + 1
    return protos


def test_binding_argument_counts_match_the_header():
    from paged_kv_cache_26_gb300._native import _SIGNATURES
    protos = header_prototypes()
    assert set(protos) == set(header_functions())
    for name, (_, args) in _SIGNATURES.items():
        assert name in protos, name
        assert len(args) == protos[name], (name, len(args), protos[name])


def test_slot_mapping_matches_oracle_and_page_example(golden_dir):
    gold = json.load(open(os.path.join(golden_dir, "block_tables.json")))
    t = gold["kasblo"]["tables"]
    tables = np.array([t["A"], t["B"] + [-1]], np.int32)
    lens = np.array([48, 18], np.int32)
    assert list(paged_kv_slot_mapping(tables, lens)) == list(oracle.slot_mapping(tables, lens, 16)) == [159, 129]
    rng = np.random.default_rng(0)
    for _ in range(20):
        B, mb = 9, 7
        tables = rng.integers(0, 500, size=(B, mb)).astype(np.int32)
        lens = rng.integers(0, mb * 16 + 1, size=B).astype(np.int32)
        assert np.array_equal(paged_kv_slot_mapping(tables, lens), oracle.slot_mapping(tables, lens, 16))


def test_slot_mapping_rejects_bad_tables():
    with pytest.raises(PagedKVError):
        paged_kv_slot_mapping(np.array([[3, -1]], np.int32), np.array([20], np.int32))
    with pytest.raises(PagedKVError):
        paged_kv_slot_mapping(np.array([[3]], np.int32), np.array([17], np.int32))


def test_allocator_lifecycle_and_scatter():
    a = BlockAllocator(64, 16, seed=1)
    s0 = a.add_seq(40)              # 3 blocks
    s1 = a.add_seq(16)              # 1 block
    assert a.num_free == 60
    tables, lens = a.block_tables([s0, s1], 4)
    assert list(lens) == [40, 16]
    assert list(tables[1, 1:]) == [-1, -1, -1]
    used = [int(x) for x in tables[tables >= 0]]
    assert len(set(used)) == 4                                    # no double allocation
    assert sorted(used) != list(range(min(used), min(used) + 4))  # scattered
    # growth: positions 40..47 stay in block 2, position 48 opens block 3
    slots = [a.append_slot(s0) for _ in range(9)]
    t2, l2 = a.block_tables([s0], 4)
    assert l2[0] == 49 and a.num_free == 59
    for pos, slot in zip(range(40, 49), slots):
        assert slot == oracle.slot_of_position(t2[0], pos, 16)
    # s1 is full: the next token takes a fresh block
    a.append_slot(s1)
    assert a.num_free == 58
    a.free_seq(s0)
    assert a.num_free == 62
    assert all(a.refcount(int(b)) == 0 for b in t2[0])
    # freed blocks are reused
    s2 = a.add_seq(62 * 16)
    assert a.num_free == 0
    with pytest.raises(PagedKVError) as e:
        a.add_seq(1)
    assert e.value.code == -5
    a.free_seq(s2)
    a.free_seq(s1)
    assert a.num_free == 64


def test_allocator_shared_prefix_refcounts():
    a = BlockAllocator(100, 16, seed=3)
    src = a.add_seq(513)
    forks = [a.fork_prefix(src, 512, 600) for _ in range(3)]
    t, _ = a.block_tables([src] + forks, 40)
    for f in range(1, 4):
        assert np.array_equal(t[f, :32], t[0, :32])
        assert len(set(t[f, 32:38]) & set(t[0, :33])) == 0
    assert all(a.refcount(int(b)) == 4 for b in t[0, :32])
    assert a.refcount(int(t[0, 32])) == 1
    a.free_seq(src)
    assert all(a.refcount(int(b)) == 3 for b in t[0, :32])
    for f in forks:
        a.free_seq(f)
    assert a.num_free == 100
    with pytest.raises(PagedKVError):
        a.fork_prefix(a.add_seq(20), 8, 30)      # prefix must be whole blocks


def test_appends_after_a_fork_never_write_shared_blocks():
    """Forks share whole blocks only, so every later append lands in a block
    whose reference count is 1."""
    a = BlockAllocator(40, 16, seed=0)
    src = a.add_seq(48)
    kids = [a.fork_prefix(src, 32, 32), a.fork_prefix(src, 48, 50), a.fork_prefix(src, 16, 16)]
    shared = set(int(b) for b in a.block_tables([src], 3)[0][0])
    for sid in [src] + kids:
        for _ in range(20):
            slot = a.append_slot(sid)
            assert slot // 16 not in shared
            assert a.refcount(slot // 16) == 1


def test_allocator_waste_below_one_block():
    a = BlockAllocator(4096, 16, seed=5)
    rng = np.random.default_rng(2)
    lens = rng.integers(1, 2000, size=50)
    ids = [a.add_seq(int(L)) for L in lens]
    t, l = a.block_tables(ids, 125)
    for row, L in zip(t, l):
        n = int((row >= 0).sum())
        assert n == oracle.blocks_needed(int(L), 16)
        assert 0 <= n * 16 - L < 16


def test_slot_mapping_multi_matches_oracle():
    rng = np.random.default_rng(5)
    B, MB, n = 7, 6, 4
    tables = np.stack([rng.permutation(40)[:MB] for _ in range(B)]).astype(np.int32)
    lens = np.array([0, 1, 3, 4, 16, 17, 96], np.int32)
    got = pkv.paged_kv_slot_mapping_multi(tables, lens, n)
    assert np.array_equal(got, oracle.slot_mapping_multi(tables, lens, n, 16))
    with pytest.raises(pkv.PagedKVError):
        pkv.paged_kv_slot_mapping_multi(tables, np.array([97] * B, np.int32), n)   # past the table


def test_attention_shape_checks_refuse_short_lengths_and_tables_before_any_launch():
    """The kernels read context_lens[b] and block_tables row b for every
    sequence b of q: shorter tensors are refused by the binding (no GPU
    needed: the check runs before any call into the library)."""
    import torch
    from paged_kv_cache_26_gb300.api import _check_attention_shapes
    q = torch.zeros(4, 8, 64, dtype=torch.float16)
    kc = torch.zeros(32, 2, 16, 64, dtype=torch.float16)
    bt = torch.zeros(4, 7, dtype=torch.int32)
    cl = torch.zeros(4, dtype=torch.int32)
    _check_attention_shapes(q, torch.empty_like(q), kc, bt, cl)
    for bad_bt, bad_cl in ((bt, cl[:3]), (bt[:3], cl), (bt[0], cl), (bt, cl.view(4, 1))):
        with pytest.raises(ValueError):
            _check_attention_shapes(q, torch.empty_like(q), kc, bad_bt, bad_cl)
    with pytest.raises(ValueError):
        _check_attention_shapes(q, torch.empty(4, 8, 32, dtype=torch.float16), kc, bt, cl)

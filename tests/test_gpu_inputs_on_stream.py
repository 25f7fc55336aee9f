"""Inputs written on the GPU right before a decode step.

The automatic path's kernels are programmatic dependents of the kernel before
them in the stream: they may start while it finishes, and read the context
lengths and block tables early, as a guess, before their grid wait.  After the
wait they read both again and rebuild anything derived from a stale guess
(include/paged_kv.h, the paragraph on programmatic dependent launches).
These tests check that contract against the fp64 oracle:

* a serving loop in which torch kernels on the same stream advance
  context_lens (add_) and store freshly allocated block ids into block_tables
  (index_put_) immediately before every paged_decode_step, with the GPU kept
  behind the host so that the launches queue back to back;
* the self-test entry point whose prologues read deliberately stale lengths
  and tables: the result must be the real inputs' result, bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_26_gb300 as pkv
import workloads as wl
from paged_kv_cache_26_gb300 import build as pkv_build
from parity_helpers import assert_close, bits, oracle_caches, oracle_rows, widen_out

pytestmark = pytest.mark.gpu

BS = 16


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv_build.build()


def _growing_batch(seed, B, Hq, Hkv, D, steps, lo, hi):
    """Initial lengths, a pool with room for `steps` more tokens per sequence,
    initial tables from a seeded scattered placement, and the blocks each
    step's growth will take (popped from the same permutation).  Slots not
    holding one of the first L0 - 1 tokens are NaN."""
    rng = np.random.default_rng(seed)
    L0 = rng.integers(lo, hi + 1, size=B).astype(np.int64)
    need = sum(-(-(int(L) + steps) // BS) for L in L0)
    nb = need + 8
    perm = list(rng.permutation(nb))
    mb = max(-(-(int(L) + steps) // BS) for L in L0)
    tables = np.full((B, mb), -1, np.int32)
    for b in range(B):
        for j in range(-(-int(L0[b]) // BS)):
            tables[b, j] = perm.pop()
    g = torch.Generator(device="cuda").manual_seed(seed)
    kc = torch.randn(nb, Hkv, BS, D, generator=g, device="cuda").to(torch.bfloat16)
    vc = torch.randn(nb, Hkv, BS, D, generator=g, device="cuda").to(torch.bfloat16)
    valid = torch.zeros(nb, BS, dtype=torch.bool)
    for b in range(B):
        for t in range(int(L0[b]) - 1):
            valid[tables[b, t // BS], t % BS] = True
    nan_mask = (~valid).to("cuda")[:, None, :, None].expand_as(kc)
    kc[nan_mask] = float("nan")
    vc[nan_mask] = float("nan")
    # The growth schedule: at step s sequence b holds L0[b] + s tokens; its
    # new token sits at position L0[b] + s - 1 and needs a fresh block when
    # that position starts one.
    grow = []
    for s in range(steps):
        new = []
        for b in range(B):
            pos = int(L0[b]) + s - 1
            if pos % BS == 0 and tables[b, pos // BS] < 0:
                new.append((b, pos // BS, perm.pop()))
                tables[b, pos // BS] = new[-1][2]
        grow.append(new)
    # tables now holds the final state; rebuild the initial one for the GPU
    init = tables.copy()
    for new in grow:
        for b, j, _ in new:
            init[b, j] = -1
    q = torch.randn(steps, B, Hq, D, generator=g, device="cuda").to(torch.bfloat16)
    kn = torch.randn(steps, B, Hkv, D, generator=g, device="cuda").to(torch.bfloat16)
    vn = torch.randn(steps, B, Hkv, D, generator=g, device="cuda").to(torch.bfloat16)
    return L0, init, grow, kc, vc, q, kn, vn


def test_lengths_and_tables_written_on_stream_right_before_each_step():
    B, Hq, Hkv, D, steps = 8, 32, 8, 128, 200
    scale = D ** -0.5
    L0, init, grow, kc, vc, q, kn, vn = _growing_batch(7, B, Hq, Hkv, D, steps, 100, 400)
    kc0, vc0 = bits(kc), bits(vc)
    dev = torch.device("cuda")
    bt = torch.from_numpy(init).to(dev)
    cl = torch.from_numpy((L0 - 1).astype(np.int32)).to(dev)
    # each step's table writes as device tensors, uploaded before the loop
    upd = [None if not new else tuple(torch.tensor(c, dtype=torch.int64 if i < 2 else torch.int32, device=dev)
                                      for i, c in enumerate(zip(*new)))
           for new in grow]
    out = torch.empty(steps, B, Hq, D, dtype=torch.bfloat16, device=dev)
    ws = pkv.make_workspace(q[0], kc, bt)
    assert pkv.paged_decode_resolve_splits(q[0], kc, bt) == 0  # the persistent, programmatic path
    torch.cuda.synchronize()
    for s in range(steps):
        if s % 25 == 0:
            torch.cuda._sleep(20_000_000)  # keep the GPU behind the host: launches queue back to back
        # alternate which input is written last before the step
        if s % 2 == 0:
            if upd[s] is not None:
                bt.index_put_((upd[s][0], upd[s][1]), upd[s][2])
            cl.add_(1)
        else:
            cl.add_(1)
            if upd[s] is not None:
                bt.index_put_((upd[s][0], upd[s][1]), upd[s][2])
        pkv.paged_decode_step(q[s], kn[s], vn[s], kc, vc, bt, cl, scale, out=out[s], workspace=ws)
    pkv.paged_kv_check_status()
    got = widen_out(out, "bf16")
    gk, gv = bits(kc), bits(vc)
    assert np.array_equal(cl.cpu().numpy(), L0 + steps - 1)

    # The oracle replays the same steps: tables grow, each token is stored at
    # position L - 1, then every (sequence, query head) row attends.
    tables = init.copy()
    rk, rv = kc0, vc0
    qb, knb, vnb = bits(q), bits(kn), bits(vn)
    rows = [(b, h) for b in range(B) for h in range(Hq)]
    for s in range(steps):
        for b, j, blk in grow[s]:
            tables[b, j] = blk
        lens = (L0 + s).astype(np.int32)
        slots = oracle.slot_mapping(tables, lens, BS)
        rk, rv = oracle.kv_append(rk, rv, knb[s], vnb[s], slots, BS)
        ref = oracle.decode_attention_rows(qb[s], rk, rv, tables, lens, scale, "bf16", BS, rows)
        assert_close(np.stack([got[s, b, h] for b, h in rows]), ref, f"step {s}")
    assert np.array_equal(gk, rk), "K appends differ from the oracle"
    assert np.array_equal(gv, rv), "V appends differ from the oracle"
    assert np.array_equal(bt.cpu().numpy(), tables)


def _stale_case(seed):
    spec = wl.LLAMA3_8B.replace(name="stale", batch=24, lengths=("uniform", 1, 900))
    w = wl.generate(spec, seed=seed, device="cuda")
    return w


@pytest.mark.parametrize("publish", [True, False], ids=["published", "merge_rechecks"])
@pytest.mark.parametrize("kind", ["lengths_and_tables", "tables_only", "garbage"])
def test_stale_prologue_inputs_are_rebuilt_after_the_wait(kind, publish):
    w = _stale_case(11)
    dev = torch.device("cuda")
    rk, rv = oracle_caches(w)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    rng = np.random.default_rng(5)
    if kind == "lengths_and_tables":
        stale_cl = np.maximum(w.context_lens - rng.integers(0, 40, w.spec.batch), 0).astype(np.int32)
        stale_bt = np.roll(w.block_tables, 1, axis=0)
    elif kind == "tables_only":
        stale_cl = w.context_lens.copy()
        stale_bt = w.block_tables.copy()
        stale_bt[stale_bt >= 0] = rng.permutation(stale_bt[stale_bt >= 0])
    else:  # lengths at the table's capacity, block ids all outside the pool: nothing may be flagged
        stale_cl = np.full_like(w.context_lens, w.max_blocks * BS)
        stale_bt = np.full_like(w.block_tables, w.num_blocks + 5)
    kc, vc = w.k_cache[0].clone(), w.v_cache[0].clone()
    out = pkv.paged_kv_selftest_stale_prologue(
        w.q[0], w.k_new[0], w.v_new[0], kc, vc, bt, cl, torch.from_numpy(stale_bt).to(dev),
        torch.from_numpy(stale_cl).to(dev), w.scale, publish=publish)
    pkv.paged_kv_check_status()  # raises if a stale value was flagged
    assert np.array_equal(bits(kc), rk) and np.array_equal(bits(vc), rv)
    rows = [(b, h) for b in range(w.spec.batch) for h in range(w.spec.num_q_heads)]
    gpu = widen_out(out, w.spec.dtype)
    assert_close(np.stack([gpu[b, h] for b, h in rows]), oracle_rows(w, rk, rv, rows), f"stale {kind}")
    # bit for bit what paged_decode_step gives on the real inputs
    kc2, vc2 = w.k_cache[0].clone(), w.v_cache[0].clone()
    ref = pkv.paged_decode_step(w.q[0], w.k_new[0], w.v_new[0], kc2, vc2, bt, cl, w.scale)
    pkv.paged_kv_check_status()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))

"""paged_decode_attention_no_alloc: attention for callers that cannot allocate
device memory while they run (plugin hosts that forbid allocation during
enqueue, processes whose device memory another allocator already holds,
latency paths that cannot take cudaMalloc's implicit synchronisation).  Its
scratch is a fixed array inside the library, so the call allocates nothing.

This file is named to be collected last: if it fails, a run that stops at the
first failure has already run every other test.  It also passes on its own in
a fresh process (the first call on the device sets up the array's address).
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_26_gb300 as pkv
import workloads as wl
from paged_kv_cache_26_gb300 import build as pkv_build
from paged_kv_cache_26_gb300._native import PkvDims, lib
from parity_helpers import ATOL, RTOL, assert_close, oracle_caches, oracle_rows, widen_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv_build.build()


def _prepared(spec, seed, with_oracle=False):
    """A workload on the GPU with this step's token already appended, and
    (with_oracle) the oracle's caches after its own append of the same token,
    taken from the bits before the GPU append."""
    dev = torch.device("cuda")
    w = wl.generate(spec, seed=seed, device=dev)
    ref_caches = oracle_caches(w) if with_oracle else None
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    slots = torch.from_numpy(pkv.paged_kv_slot_mapping(w.block_tables, w.context_lens)).to(dev)
    pkv.paged_kv_append(w.k_new[0], w.v_new[0], slots, w.k_cache[0], w.v_cache[0])
    return (w, bt, cl, ref_caches) if with_oracle else (w, bt, cl)


def _call_no_alloc(w, bt, cl, out, num_splits):
    """Straight through the C ABI."""
    s = w.spec
    dims = PkvDims(num_seqs=s.batch, num_q_heads=s.num_q_heads, num_kv_heads=s.num_kv_heads, head_dim=s.head_dim,
                   block_size=s.block_size, num_blocks=w.num_blocks, max_blocks_per_seq=w.max_blocks,
                   dtype=0 if s.dtype == "fp16" else 1)
    P = ctypes.c_void_p
    return lib().paged_decode_attention_no_alloc(
        P(w.q[0].data_ptr()), P(w.k_cache[0].data_ptr()), P(w.v_cache[0].data_ptr()), P(bt.data_ptr()),
        P(cl.data_ptr()), ctypes.c_float(w.scale), P(out.data_ptr()), num_splits, ctypes.byref(dims),
        P(torch.cuda.current_stream().cuda_stream))


def _close(a, b):
    a, b = a.float().cpu().numpy(), b.float().cpu().numpy()
    assert np.all(np.isfinite(a))
    assert np.all(np.abs(a - b) <= ATOL + RTOL * np.abs(b)), float(np.abs(a - b).max())


def test_no_alloc_matches_the_oracle_and_the_workspace_entry_point_on_two_calls_in_a_row():
    # Two different batches back to back: the second call reuses the scratch the
    # first one filled, and must not see any of it.  Every output row is
    # compared with the fp64 oracle and with paged_decode_attention.
    cases = [(wl.LLAMA3_8B.replace(batch=16), 0, 0), (wl.LONG_CTX.replace(batch=2), 1, 64)]
    for spec, seed, splits in cases:
        w, bt, cl, (rk, rv) = _prepared(spec, seed, with_oracle=True)
        ref = pkv.paged_decode_attention(w.q[0], w.k_cache[0], w.v_cache[0], bt, cl, w.scale)
        out = torch.empty_like(w.q[0])
        assert _call_no_alloc(w, bt, cl, out, splits) == 0, lib().paged_kv_last_error()
        pkv.paged_kv_check_status()
        _close(out, ref)
        B, H, D = spec.batch, spec.num_q_heads, spec.head_dim
        rows = [(b, h) for b in range(B) for h in range(H)]
        gpu = widen_out(out, spec.dtype)
        assert_close(np.stack([gpu[b, h] for b, h in rows]), oracle_rows(w, rk, rv, rows),
                     f"no_alloc {spec.name} splits={splits}")
    # and the same batch twice: identical bits
    w, bt, cl = _prepared(wl.LLAMA3_8B.replace(batch=8), 2)
    a, b = torch.empty_like(w.q[0]), torch.empty_like(w.q[0])
    assert _call_no_alloc(w, bt, cl, a, 0) == 0
    assert _call_no_alloc(w, bt, cl, b, 0) == 0
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_no_alloc_python_wrapper_matches_the_oracle_and_checks_shapes():
    spec = wl.LLAMA70B_TAIL.replace(batch=12, lengths=("lognormal", 300.0, 1.0, 1, 1500), shared_prefix=(3, 64))
    w, bt, cl, (rk, rv) = _prepared(spec, 4, with_oracle=True)
    out = torch.empty_like(w.q[0])
    pkv.paged_decode_attention_no_alloc(w.q[0], w.k_cache[0], w.v_cache[0], bt, cl, w.scale, out)
    pkv.paged_kv_check_status()
    rows = [(b, h) for b in range(spec.batch) for h in range(spec.num_q_heads)]
    gpu = widen_out(out, spec.dtype)
    assert_close(np.stack([gpu[b, h] for b, h in rows]), oracle_rows(w, rk, rv, rows), "no_alloc wrapper")
    # a context_lens or block_tables shorter than the batch is refused before any launch
    with pytest.raises(ValueError):
        pkv.paged_decode_attention_no_alloc(w.q[0], w.k_cache[0], w.v_cache[0], bt, cl[:-1], w.scale, out)
    with pytest.raises(ValueError):
        pkv.paged_decode_attention_no_alloc(w.q[0], w.k_cache[0], w.v_cache[0], bt[:-1], cl, w.scale, out)


def test_no_alloc_rejects_a_batch_beyond_its_scratch():
    w, bt, cl = _prepared(wl.LLAMA3_8B.replace(batch=64), 3)
    out = torch.empty_like(w.q[0])
    # 64 sequences x 32 heads x 256 one-block splits x 129 floats: ~270 MB > 16 MiB
    rc = _call_no_alloc(w, bt, cl, out, 256)
    assert rc == -1
    msg = lib().paged_kv_last_error().decode()
    assert "static scratch holds 16777216" in msg

"""GPU parity of multi-token paged decode (q_len new tokens per sequence,
causal among them) against the fp64 oracle.

Append: the pool after the q_len-token append equals the oracle's bit for bit.
Attention: |gpu - ref| <= 2e-3 + 1e-2 |ref| elementwise, the bound of the
one-token path (same arithmetic: fp32 accumulation, rounded softmax weights).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_26_gb300 as pkv
import workloads as wl
from paged_kv_cache_26_gb300 import build as pkv_build
from parity_helpers import assert_close, bits, widen_out

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv_build.build()


def run_multi(w, m, layer=0, num_splits=0, fused=True, tensor_cores=False):
    kc = w.k_cache[layer].to(DEV, copy=True)
    vc = w.v_cache[layer].to(DEV, copy=True)
    q, kn, vn = (t[layer].to(DEV) for t in (m.q, m.k_new, m.v_new))
    bt = torch.from_numpy(w.block_tables).to(DEV)
    cl = torch.from_numpy(w.context_lens).to(DEV)
    if fused:
        out = pkv.paged_decode_step_multi(q, kn, vn, kc, vc, bt, cl, w.scale, num_splits=num_splits,
                                          tensor_cores=tensor_cores)
    else:
        slots = pkv.paged_kv_slot_mapping_multi(w.block_tables, w.context_lens, m.q_len).reshape(-1)
        B, n = kn.shape[:2]
        pkv.paged_kv_append(kn.reshape(B * n, *kn.shape[2:]), vn.reshape(B * n, *vn.shape[2:]),
                            torch.from_numpy(slots).to(DEV), kc, vc)
        out = pkv.paged_decode_attention_multi(q, kc, vc, bt, cl, w.scale, num_splits=num_splits)
    pkv.paged_kv_check_status()
    return out.cpu(), kc.cpu(), vc.cpu()


def oracle_multi_caches(w, m, layer=0):
    slots = oracle.slot_mapping_multi(w.block_tables, w.context_lens, m.q_len, w.spec.block_size).reshape(-1)
    kn, vn = bits(m.k_new[layer]), bits(m.v_new[layer])
    B, n = kn.shape[:2]
    return oracle.kv_append(bits(w.k_cache[layer]), bits(w.v_cache[layer]), kn.reshape(B * n, *kn.shape[2:]),
                            vn.reshape(B * n, *vn.shape[2:]), slots, w.spec.block_size)


def check_multi(w, m, layer=0, num_splits=0, rows=None, fused=True, tensor_cores=False):
    out, kc, vc = run_multi(w, m, layer, num_splits, fused, tensor_cores)
    rk, rv = oracle_multi_caches(w, m, layer)
    assert np.array_equal(bits(kc), rk), "K append differs from the oracle"
    assert np.array_equal(bits(vc), rv), "V append differs from the oracle"
    B, n, H = w.spec.batch, m.q_len, w.spec.num_q_heads
    if rows is None:
        rows = [(b, i, h) for b in range(B) for i in range(n) for h in range(H)]
    ref = oracle.decode_attention_multi(bits(m.q[layer]), rk, rv, w.block_tables, w.context_lens, n, w.scale,
                                        w.spec.dtype, w.spec.block_size, rows=rows)
    gpu = widen_out(out, w.spec.dtype)
    assert_close(np.stack([gpu[b, i, h] for b, i, h in rows]), ref,
                 f"multi {w.spec.name} q_len={n} splits={num_splits} fused={fused}")
    return out


CASES = [
    (wl.TINY, 4),                                                                           # D 64, fp16, g 4
    (wl.LLAMA3_8B.replace(name="llama8b_small", batch=5, lengths=("uniform", 1, 700)), 2),  # 8 rows, 1 warp
    (wl.LLAMA3_8B.replace(name="llama8b_small", batch=5, lengths=("uniform", 1, 700)), 3),  # 12 rows, padding
    (wl.LLAMA3_8B.replace(name="llama8b_small", batch=4, lengths=("uniform", 1, 700)), 8),  # 32 rows, 4 warps
    (wl.LLAMA70B_TAIL.replace(name="70b_small", batch=6, lengths=("lognormal", 200.0, 1.0, 1, 900),
                              shared_prefix=(2, 64)), 8),                                   # g 8: 64 rows, 8 warps
    (wl.MHA_7B_B16.replace(name="mha_small", batch=3, lengths=("constant", 333), num_layers=1), 5),  # g 1
]


@pytest.mark.parametrize("splits", [1, 3, 0])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0].name}-q{c[1]}")
def test_multi_every_output(case, splits):
    spec, n = case
    w, m = wl.generate_multi(spec, n, seed=7)
    check_multi(w, m, num_splits=splits)


def test_multi_separate_append_matches_fused():
    w, m = wl.generate_multi(CASES[3][0], 8, seed=2)
    a = check_multi(w, m, fused=True)
    b = check_multi(w, m, fused=False)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("n", [1, 4, 8])
def test_multi_edge_lengths(n):
    # shorter than q_len, exactly q_len, new tokens across a block boundary, empty
    lens = (1, 2, n, 18, 16, 17, 0, 33, 512, 513)
    spec = wl.LLAMA3_8B.replace(name="custom", batch=len(lens), lengths=("fixed", lens), pool=("factor", 1.5),
                                num_q_heads=8, num_kv_heads=2)
    w, m = wl.generate_multi(spec, n, seed=3)
    for splits in (1, 2, 0):
        out = check_multi(w, m, num_splits=splits)
        assert torch.all(out[6] == 0)                      # empty context: zero rows
        if n > 1:
            assert torch.all(out[0, :n - 1] == 0)          # tokens before position 0: zero rows


def test_multi_q_len_one_equals_single_token_step():
    w, m = wl.generate_multi(wl.LLAMA3_8B.replace(name="l8", batch=6, lengths=("uniform", 1, 300)), 1, seed=4)
    out = run_multi(w, m)[0]
    dev = torch.device(DEV)
    kc, vc = w.k_cache[0].to(dev, copy=True), w.v_cache[0].to(dev, copy=True)
    bt, cl = torch.from_numpy(w.block_tables).to(dev), torch.from_numpy(w.context_lens).to(dev)
    one = pkv.paged_decode_step(m.q[0][:, 0].to(dev), m.k_new[0][:, 0].to(dev), m.v_new[0][:, 0].to(dev), kc, vc,
                                bt, cl, w.scale, num_splits=1)
    ref = widen_out(one.cpu(), "bf16")
    assert_close(widen_out(out[:, 0], "bf16"), ref, "q_len 1 vs one-token step")


def test_multi_llama3_8b_full_sampled():
    w, m = wl.generate_multi(wl.LLAMA3_8B, 4, seed=0, device=DEV)
    rng = np.random.default_rng(0)
    rows = sorted({(int(rng.integers(64)), int(rng.integers(4)), int(rng.integers(32))) for _ in range(96)}
                  | {(int(np.argmax(w.context_lens)), 3, 0), (int(np.argmin(w.context_lens)), 0, 31)})
    check_multi(w, m, rows=rows)


@pytest.mark.parametrize("splits", [1, 0])
def test_multi_step_from_host_chained_matches_device_calls(splits):
    """Multi-token host-buffer steps issued back to back through one device
    staging area (kernel copies in and out, pinned buffers), each with its own
    inputs and output: outputs and final caches equal those of the same steps
    run from device tensors."""
    w, m = wl.generate_multi(CASES[3][0], 4, seed=11)
    dev = torch.device(DEV)
    g = torch.Generator().manual_seed(4)
    keys = ["q", "k_new", "v_new", "block_tables", "context_lens"]
    steps = [{"q": torch.randn(m.q[0].shape, generator=g).bfloat16(),
              "k_new": torch.randn(m.k_new[0].shape, generator=g).bfloat16(),
              "v_new": torch.randn(m.v_new[0].shape, generator=g).bfloat16(),
              "block_tables": torch.from_numpy(w.block_tables).clone(),
              "context_lens": torch.from_numpy(w.context_lens).clone()} for _ in range(3)]
    kc_ref, vc_ref = w.k_cache[0].to(dev, copy=True), w.v_cache[0].to(dev, copy=True)
    ref = []
    for st in steps:
        d = {k: v.to(dev) for k, v in st.items()}
        ref.append(pkv.paged_decode_step_multi(d["q"], d["k_new"], d["v_new"], kc_ref, vc_ref, d["block_tables"],
                                               d["context_lens"], w.scale, num_splits=splits).cpu())
    kc, vc = w.k_cache[0].to(dev, copy=True), w.v_cache[0].to(dev, copy=True)
    devb = {k: torch.empty_like(steps[0][k], device=dev) for k in keys}
    devb["out"] = torch.empty_like(steps[0]["q"], device=dev)
    hosts = [{**{k: st[k].contiguous().pin_memory() for k in keys},
              "out": torch.full_like(st["q"], float("nan")).pin_memory()} for st in steps]
    for h in hosts:
        pkv.paged_decode_step_multi_from_host(h, devb, kc, vc, w.scale, num_splits=splits)
    torch.cuda.synchronize()
    pkv.paged_kv_check_status()
    for h, r in zip(hosts, ref):
        assert torch.equal(h["out"].view(torch.int16), r.view(torch.int16))
    assert torch.equal(kc.view(torch.int16), kc_ref.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), vc_ref.view(torch.int16))


def test_multi_invalid_arguments_are_rejected():
    dev = torch.device(DEV)
    kc = torch.zeros(8, 2, 16, 128, dtype=torch.bfloat16, device=dev)
    bt = torch.zeros(2, 1, dtype=torch.int32, device=dev)
    cl = torch.ones(2, dtype=torch.int32, device=dev)
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_decode_attention_multi(torch.zeros(2, 9, 8, 128, dtype=torch.bfloat16, device=dev), kc, kc, bt,
                                         cl, 0.1)
    assert e.value.code == -2
    with pytest.raises(ValueError):
        pkv.paged_decode_attention_multi(torch.zeros(2, 8, 128, dtype=torch.bfloat16, device=dev), kc, kc, bt, cl,
                                         0.1)


# ---- the tensor-core (tcgen05) kernel: 64 query rows per KV head, head_dim 128

TC_70B_SMALL = wl.LLAMA70B_TAIL.replace(name="70b_small", batch=6, lengths=("lognormal", 200.0, 1.0, 1, 900),
                                        shared_prefix=(2, 64))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_multi_tensor_cores_every_output(dtype, splits):
    w, m = wl.generate_multi(TC_70B_SMALL.replace(dtype=dtype), 8, seed=7)
    check_multi(w, m, num_splits=splits, tensor_cores=True)


def test_multi_tensor_cores_edge_lengths():
    # empty, shorter than q_len, exactly q_len, new tokens across block boundaries,
    # a split boundary (512 / 513 with two splits)
    lens = (1, 2, 8, 18, 16, 17, 0, 33, 512, 513)
    spec = wl.LLAMA3_8B.replace(name="custom", batch=len(lens), lengths=("fixed", lens), pool=("factor", 1.5),
                                num_q_heads=16, num_kv_heads=2)
    w, m = wl.generate_multi(spec, 8, seed=3)
    for splits in (1, 2, 0):
        out = check_multi(w, m, num_splits=splits, tensor_cores=True)
        assert torch.all(out[6] == 0)              # empty context: zero rows
        assert torch.all(out[0, :7] == 0)          # tokens before position 0: zero rows


def test_multi_tensor_cores_llama70b_full_sampled():
    w, m = wl.generate_multi(wl.LLAMA70B_TAIL, 8, seed=0, device=DEV)
    rng = np.random.default_rng(1)
    rows = sorted({(int(rng.integers(256)), int(rng.integers(8)), int(rng.integers(64))) for _ in range(96)}
                  | {(int(np.argmax(w.context_lens)), 7, 0), (int(np.argmin(w.context_lens)), 0, 63)})
    check_multi(w, m, rows=rows, tensor_cores=True)


def test_multi_tensor_cores_reject_other_shapes():
    w, m = wl.generate_multi(TC_70B_SMALL, 4, seed=7)     # 32 rows per KV head
    with pytest.raises(pkv.PagedKVError):
        run_multi(w, m, tensor_cores=True)

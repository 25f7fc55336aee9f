"""GPU parity of the E4M3 (FP8) KV cache path against the fp64 oracle.

Append: the quantised codes are compared bit for bit over the whole pool
(untouched NaN-code slots included).  Attention: the oracle attends over the
dequantised pool (code value * the KV head's scale) in float64; the GPU output
must be within |gpu - ref| <= 2e-3 + 1e-2 |ref| elementwise, the same bound as
the fp16/bf16 path (the GPU's E4M3 -> fp16 conversion is exact, so the error
budget is the same: fp32 accumulation and the rounding of the softmax weights).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_26_gb300 as pkv
import workloads as wl
from paged_kv_cache_26_gb300 import build as pkv_build
from parity_helpers import assert_close, bits, sample_rows, widen_out

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv_build.build()


def run_fp8(w, f8, layer=0, fused=True):
    """One decode step over the E4M3 pool through the C ABI.  Returns (out,
    k_codes, v_codes) on the CPU; the workload's tensors are not modified."""
    kc = f8.k_cache[layer].to(DEV, copy=True)
    vc = f8.v_cache[layer].to(DEV, copy=True)
    ks, vs = f8.k_scale[layer].to(DEV), f8.v_scale[layer].to(DEV)
    q, kn, vn = (t[layer].to(DEV) for t in (w.q, w.k_new, w.v_new))
    bt = torch.from_numpy(w.block_tables).to(DEV)
    cl = torch.from_numpy(w.context_lens).to(DEV)
    if fused:
        out = pkv.paged_decode_step_fp8(q, kn, vn, kc, vc, ks, vs, bt, cl, w.scale)
    else:
        slots = torch.from_numpy(pkv.paged_kv_slot_mapping(w.block_tables, w.context_lens)).to(DEV)
        pkv.paged_kv_append_fp8(kn, vn, slots, kc, vc, ks, vs)
        out = pkv.paged_decode_attention_fp8(q, kc, vc, ks, vs, bt, cl, w.scale)
    pkv.paged_kv_check_status()
    return out.cpu(), kc.cpu().numpy(), vc.cpu().numpy()


def oracle_fp8_caches(w, f8, layer=0):
    slots = oracle.slot_mapping(w.block_tables, w.context_lens, w.spec.block_size)
    return oracle.kv_append_fp8(f8.k_cache[layer].cpu().numpy(), f8.v_cache[layer].cpu().numpy(),
                                bits(w.k_new[layer]), bits(w.v_new[layer]), slots, w.spec.block_size,
                                f8.k_scale[layer].cpu().numpy(), f8.v_scale[layer].cpu().numpy(), w.spec.dtype)


def check_fp8(w, f8, layer=0, rows=None, fused=True):
    out, kc, vc = run_fp8(w, f8, layer, fused)
    rk, rv = oracle_fp8_caches(w, f8, layer)
    assert np.array_equal(kc, rk), "K codes differ from the oracle's quantised append"
    assert np.array_equal(vc, rv), "V codes differ from the oracle's quantised append"
    B, H = w.spec.batch, w.spec.num_q_heads
    if rows is None:
        rows = [(b, h) for b in range(B) for h in range(H)]
    scales = (f8.k_scale[layer].cpu().numpy(), f8.v_scale[layer].cpu().numpy())
    ref = oracle.decode_attention_rows(bits(w.q[layer]), rk, rv, w.block_tables, w.context_lens, w.scale,
                                       w.spec.dtype, w.spec.block_size, rows, kv_scales=scales)
    gpu = widen_out(out, w.spec.dtype)
    assert_close(np.stack([gpu[b, h] for b, h in rows]), ref, f"fp8 {w.spec.name} fused={fused}")
    return out


REDUCED = [
    wl.TINY.replace(name="tiny_d128", head_dim=128, pool=("factor", 1.5)),
    wl.TINY.replace(name="tiny_d128_bf16_mqa", head_dim=128, num_kv_heads=1, dtype="bf16", pool=("factor", 2.0)),
    wl.LLAMA3_8B.replace(name="llama8b_small", batch=6, lengths=("uniform", 1, 700)),
    wl.MHA_7B_B16.replace(name="mha_small", batch=3, lengths=("constant", 333), num_layers=2),
    wl.LLAMA70B_TAIL.replace(name="70b_small", batch=24, lengths=("lognormal", 200.0, 1.0, 1, 900),
                             shared_prefix=(4, 64)),
    wl.LONG_CTX.replace(name="long_small", batch=2, lengths=("constant", 2100)),
]


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("spec", REDUCED, ids=lambda s: s.name)
def test_fp8_reduced_configs_every_output(spec, fused):
    w = wl.generate(spec, seed=5)
    f8 = wl.fp8_caches(w, seed=5)
    for layer in range(len(w.q)):
        check_fp8(w, f8, layer, fused=fused)


def test_fp8_llama3_8b_full_every_output():
    w = wl.generate(wl.LLAMA3_8B, seed=0, device=DEV)
    check_fp8(w, wl.fp8_caches(w))


@pytest.mark.parametrize("spec", [wl.LLAMA70B_TAIL, wl.LONG_CTX, wl.MHA_7B_B64], ids=lambda s: s.name)
def test_fp8_full_sampled(spec):
    w = wl.generate(spec, seed=0, device=DEV, layers=1)
    rows = sample_rows(w, 48)
    if spec.spike_logit is not None:
        rows = sorted(set(rows + [(b, 0) for b in range(spec.batch)]))
    check_fp8(w, wl.fp8_caches(w), rows=rows)


@pytest.mark.parametrize("lens", [(1,), (5, 0, 7), (16,) * 3, (17, 1, 33), (4096, 1, 1, 1), (0, 0)])
def test_fp8_edge_lengths(lens):
    spec = wl.LLAMA3_8B.replace(name="custom", batch=len(lens), lengths=("fixed", tuple(lens)),
                                pool=("factor", 1.5), num_q_heads=16, num_kv_heads=2)
    w = wl.generate(spec, seed=2)
    check_fp8(w, wl.fp8_caches(w, seed=2))


def test_fp8_maximum_batch():
    spec = wl.LLAMA3_8B.replace(name="b2048", batch=2048, lengths=("uniform", 1, 40), num_q_heads=8,
                                num_kv_heads=2)
    w = wl.generate(spec, seed=4, device=DEV)
    check_fp8(w, wl.fp8_caches(w, seed=4), rows=sample_rows(w, 64))


def test_fp8_fused_and_separate_give_identical_bits():
    w = wl.generate(REDUCED[2], seed=9)
    f8 = wl.fp8_caches(w, seed=9)
    a = run_fp8(w, f8, fused=True)
    b = run_fp8(w, f8, fused=False)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])


def test_fp8_step_from_host_chained_matches_device_calls():
    """Host-buffer E4M3 steps issued back to back through one device staging
    area (kernel copies in and out, pinned buffers), each with its own inputs
    and output: outputs and final codes equal those of the same steps run
    from device tensors."""
    w = wl.generate(wl.LLAMA3_8B.replace(batch=7), seed=9)
    f8 = wl.fp8_caches(w, seed=9)
    dev = torch.device(DEV)
    ks, vs = f8.k_scale[0].to(dev), f8.v_scale[0].to(dev)
    g = torch.Generator().manual_seed(2)
    keys = ["q", "k_new", "v_new", "block_tables", "context_lens"]
    steps = [{"q": torch.randn(w.q[0].shape, generator=g).bfloat16(),
              "k_new": torch.randn(w.k_new[0].shape, generator=g).bfloat16(),
              "v_new": torch.randn(w.v_new[0].shape, generator=g).bfloat16(),
              "block_tables": torch.from_numpy(w.block_tables).clone(),
              "context_lens": torch.from_numpy(w.context_lens).clone()} for _ in range(3)]
    kc_ref, vc_ref = f8.k_cache[0].to(dev, copy=True), f8.v_cache[0].to(dev, copy=True)
    ref = []
    for st in steps:
        d = {k: v.to(dev) for k, v in st.items()}
        ref.append(pkv.paged_decode_step_fp8(d["q"], d["k_new"], d["v_new"], kc_ref, vc_ref, ks, vs,
                                             d["block_tables"], d["context_lens"], w.scale).cpu())
    kc, vc = f8.k_cache[0].to(dev, copy=True), f8.v_cache[0].to(dev, copy=True)
    devb = {k: torch.empty_like(steps[0][k], device=dev) for k in keys}
    devb["out"] = torch.empty_like(steps[0]["q"], device=dev)
    hosts = [{**{k: st[k].contiguous().pin_memory() for k in keys},
              "out": torch.full_like(st["q"], float("nan")).pin_memory()} for st in steps]
    need = pkv.paged_decode_workspace_bytes(devb["q"], w.k_cache[0], devb["block_tables"])
    ws = torch.zeros(need, dtype=torch.uint8, device=dev)
    for h in hosts:
        pkv.paged_decode_step_fp8_from_host(h, devb, kc, vc, ks, vs, w.scale, ws)
    torch.cuda.synchronize()
    pkv.paged_kv_check_status()
    for h, r in zip(hosts, ref):
        assert torch.equal(h["out"].view(torch.int16), r.view(torch.int16))
    assert torch.equal(kc, kc_ref) and torch.equal(vc, vc_ref)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_fp8_append_rounding_saturation_and_skips(dtype):
    """Values on both sides of E4M3's range: zeros, subnormal codes, ties,
    saturation past 448 * scale, negative zero; slot -1 is skipped."""
    g = torch.Generator().manual_seed(0)
    Hk, D, NB, n = 2, 128, 6, 40
    mag = torch.exp(torch.empty(n, Hk, D).uniform_(-14, 9, generator=g))
    sign = torch.where(torch.rand(n, Hk, D, generator=g) < 0.5, -1.0, 1.0)
    kn = (mag * sign).to(dtype)
    vn = (torch.randn(n, Hk, D, generator=g) * 3).to(dtype)
    kn[0, 0, :4] = torch.tensor([0.0, -0.0, 448 * 0.5, 464 * 0.5])
    ks = torch.tensor([0.5, 0.03125], dtype=torch.float32)
    vs = torch.tensor([0.011, 0.0173], dtype=torch.float32)
    slots = np.random.default_rng(1).permutation(NB * 16)[:n].astype(np.int32)
    slots[3] = -1
    kc = torch.full((NB, Hk, 16, D), 0x7F, dtype=torch.uint8)
    vc = kc.clone()
    rk, rv = oracle.kv_append_fp8(kc.numpy(), vc.numpy(), bits(kn), bits(vn), slots, 16, ks.numpy(), vs.numpy(),
                                  "bf16" if dtype == torch.bfloat16 else "fp16")
    kd, vd = kc.to(DEV), vc.to(DEV)
    pkv.paged_kv_append_fp8(kn.to(DEV), vn.to(DEV), torch.from_numpy(slots).to(DEV), kd, vd, ks.to(DEV),
                            vs.to(DEV))
    pkv.paged_kv_check_status()
    assert np.array_equal(kd.cpu().numpy(), rk)
    assert np.array_equal(vd.cpu().numpy(), rv)
    codes = rk[slots[0] // 16, 0, slots[0] % 16, :4]
    assert list(codes) == [0x00, 0x80, 0x7E, 0x7E]          # 0, -0, 448, 464 -> saturated to 448
    assert (rk == 0x7E).any() and (rk == 0xFE).any()       # saturation on both signs
    assert (((rk & 0x78) == 0) & ((rk & 0x07) != 0)).any()  # nonzero subnormal codes occur


def test_fp8_bf16_query_beyond_fp16_range_is_flagged():
    spec = wl.LLAMA3_8B.replace(name="qbig", batch=2, lengths=("fixed", (20, 40)), pool=("factor", 1.5))
    w = wl.generate(spec, seed=1)
    f8 = wl.fp8_caches(w, seed=1)
    w.q[0][1, 3, 5] = 1.0e5
    with pytest.raises(pkv.PagedKVError) as e:
        run_fp8(w, f8)
    assert e.value.code == -6 and "fp16 range" in str(e.value)
    pkv.paged_kv_check_status()  # cleared


def test_fp8_invalid_arguments_are_rejected():
    dev = torch.device(DEV)
    q = torch.zeros(2, 8, 64, dtype=torch.bfloat16, device=dev)
    kc = torch.zeros(4, 2, 16, 64, dtype=torch.uint8, device=dev)
    bt = torch.zeros(2, 1, dtype=torch.int32, device=dev)
    cl = torch.ones(2, dtype=torch.int32, device=dev)
    s = torch.ones(2, dtype=torch.float32, device=dev)
    with pytest.raises(pkv.PagedKVError) as e:          # head_dim 64 is not built for E4M3
        pkv.paged_decode_attention_fp8(q, kc, kc, s, s, bt, cl, 0.1)
    assert e.value.code == -2
    q = torch.zeros(2049, 8, 128, dtype=torch.bfloat16, device=dev)
    kc = torch.zeros(4, 2, 16, 128, dtype=torch.uint8, device=dev)
    bt = torch.zeros(2049, 1, dtype=torch.int32, device=dev)
    cl = torch.ones(2049, dtype=torch.int32, device=dev)
    with pytest.raises(pkv.PagedKVError) as e:          # more sequences than the shared-memory prefix holds
        pkv.paged_decode_attention_fp8(q, kc, kc, s, s, bt, cl, 0.1)
    assert e.value.code == -2
    with pytest.raises(ValueError):
        pkv.paged_decode_attention_fp8(q, kc, kc, s[:1], s, bt, cl, 0.1)
    with pytest.raises(ValueError):
        pkv.paged_decode_attention_fp8(q, kc.half(), kc, s, s, bt, cl, 0.1)

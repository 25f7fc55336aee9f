#!/usr/bin/env python
"""Decode-step benchmark for the paged KV cache.

One step = the per-token KV append plus paged decode attention (and the split
merge when the context is split) for a whole batch, on inputs resident in HBM.
Metric: achieved HBM GB/s of the step's algorithmic bytes, with decode steps/s.

Algorithmic bytes of one attention call:
    sum_b L_b * Hkv * D * 2 * sizeof(T)      K and V of every cached token
  + 2 * B * Hq * D * sizeof(T)               q read, out written
  + 4 * sum_b ceil(L_b / 16) + 4 * B          block-table entries used, context lengths
and of one append: 2 * (2 * B * Hkv * D * sizeof(T)) + 4 * B (read + write of
the new K/V rows, the slot mapping).

    python bench.py [--config llama3_8b_b64] [--steps K] [--warmup W] [--splits 0]
    python bench.py --impl reference      # the fp64 oracle on the host cores

Under torchrun each rank runs its own batch (seed + rank): the path shards by
sequence with no exchange, so scaling is weak and `value` sums all ranks' bytes
over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "paged decode attention HBM GB/s (% of ~8 TB/s roofline); decode steps/sec"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129 * 2 ** 20


# ----------------------------------------------------------------------------- bytes model

def attention_bytes(lens, batch, num_q_heads, num_kv_heads, head_dim, elem_bytes, block_size=16,
                    kv_elem_bytes=None) -> int:
    """kv_elem_bytes: bytes per cached K/V element (1 for an E4M3 pool);
    defaults to elem_bytes, the size of q / out elements."""
    kv_elem = elem_bytes if kv_elem_bytes is None else kv_elem_bytes
    lens = np.asarray(lens, np.int64)
    kv = int(lens.sum()) * num_kv_heads * head_dim * 2 * kv_elem
    q_out = 2 * batch * num_q_heads * head_dim * elem_bytes
    tables = 4 * int(((lens + block_size - 1) // block_size).sum())
    return kv + q_out + tables + 4 * batch


def append_bytes(batch, num_kv_heads, head_dim, elem_bytes, kv_elem_bytes=None) -> int:
    """New K/V rows read (elem_bytes each) and written into the pool
    (kv_elem_bytes each, default elem_bytes), plus the slot of each sequence."""
    kv_elem = elem_bytes if kv_elem_bytes is None else kv_elem_bytes
    return 2 * batch * num_kv_heads * head_dim * (elem_bytes + kv_elem) + 4 * batch


def unique_kv_bytes(w, kv_elem_bytes=2) -> int:
    """K+V bytes of distinct physical blocks read (shared prefix blocks once)."""
    s = w.spec
    n_tok = 0
    seen = set()
    for b in range(s.batch):
        L = int(w.context_lens[b])
        for j in range(-(-L // s.block_size)):
            blk = int(w.block_tables[b, j])
            if blk in seen:
                continue
            seen.add(blk)
            n_tok += min(s.block_size, L - j * s.block_size)
    return n_tok * s.num_kv_heads * s.head_dim * 2 * kv_elem_bytes


# ----------------------------------------------------------------------------- environment

def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# The sources that define the decode and merge kernels: a profile taken from
# other sources no longer describes them.
DECODE_KERNEL_SOURCES = ("paged_kv_kernels.cuh", "pkv_device.cuh")


def kernel_source_hash() -> str:
    csrc = os.path.join(ROOT, "paged_kv_cache_26_gb300", "csrc")
    h = hashlib.sha256()
    for name in DECODE_KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def ncu_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary of this
    workload, if it was captured from the current kernel sources."""
    path = os.path.join(ROOT, "profiles", f"decode_persistent_kernel_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_bytes = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not (m_hash and m_bytes) or m_hash.group(1) != kernel_source_hash():
        return None
    return float(m_bytes.group(1))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        ident = str(device_index)
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", ident], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 8:
                continue
            try:
                self.samples.append((time.time(), float(parts[1]), float(parts[2]), parts[4:]))
            except ValueError:
                continue

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        window = [s for s in self.samples if t0 - 0.15 <= s[0] <= t1 + 0.15] or self.samples
        if not window:
            return None
        reasons = sorted({name for s in window for name, v in zip(self.REASONS, s[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(s[1] for s in window), "sm_max_mhz": max(s[2] for s in window),
                "reasons": reasons, "samples": len(window)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle

def host_sample(w, seqs, layer=0, caches=None):
    """Host copies (16-bit patterns, or E4M3 codes for an fp8 pool given as
    ``caches``) of q and of the K/V blocks the listed sequences use, with their
    block tables renumbered into the copy."""
    s = w.spec
    blocks = sorted({int(x) for b in seqs for x in w.block_tables[b, :-(-int(w.context_lens[b]) // s.block_size)]})
    remap = {blk: i for i, blk in enumerate(blocks)}
    kcache, vcache = caches if caches is not None else (w.k_cache[layer], w.v_cache[layer])
    idx = torch.tensor(blocks, dtype=torch.long, device=kcache.device)

    def bits(t):
        if t.dtype == torch.uint8:
            return t.contiguous().cpu().numpy()
        return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)

    kc = bits(kcache.index_select(0, idx)) if blocks else np.zeros((0,), np.uint16)
    vc = bits(vcache.index_select(0, idx)) if blocks else np.zeros((0,), np.uint16)
    tables = np.full((len(seqs), w.block_tables.shape[1]), -1, np.int32)
    for i, b in enumerate(seqs):
        n = -(-int(w.context_lens[b]) // s.block_size)
        tables[i, :n] = [remap[int(x)] for x in w.block_tables[b, :n]]
    q = bits(w.q[layer][list(seqs)])
    return q, kc, vc, tables, w.context_lens[list(seqs)]


def oracle_rows_timed(w, sample, rows, kv_scales=None):
    import oracle
    q, kc, vc, tables, lens = sample
    t0 = time.perf_counter()
    oracle.decode_attention_rows(q, kc, vc, tables, lens, w.scale, w.spec.dtype, w.spec.block_size, rows,
                                 kv_scales=kv_scales)
    return time.perf_counter() - t0


def row_bytes(w, lens_rows, kv_elem_bytes=2) -> int:
    """Algorithmic bytes of attention for individual (sequence, query head)
    rows: each row's share of its KV head's K/V, plus its q and out."""
    s = w.spec
    g = s.group
    return sum(int(L) * s.head_dim * 2 * kv_elem_bytes / g + 2 * s.head_dim * 2 for L in lens_rows)


def cpu_baseline(w, budget_s: float, fp8=None):
    """The oracle, as it stands, over the batch's sequences in order (all query
    heads; the batch again from its start if it is done early) until about
    budget_s seconds of single-threaded CPU work.  ``fp8``: the E4M3 pool."""
    s = w.spec
    spent, done_bytes, seqs_done = 0.0, 0.0, 0
    caches = (fp8.k_cache[0], fp8.v_cache[0]) if fp8 is not None else None
    scales = (fp8.k_scale[0].cpu().numpy(), fp8.v_scale[0].cpu().numpy()) if fp8 is not None else None
    samples = {}
    while spent < budget_s:
        b = seqs_done % s.batch
        if b not in samples:
            samples[b] = host_sample(w, [b], caches=caches)
        rows = [(0, h) for h in range(s.num_q_heads)]
        spent += oracle_rows_timed(w, samples[b], rows, kv_scales=scales)
        done_bytes += row_bytes(w, [w.context_lens[b]] * s.num_q_heads, 1 if fp8 is not None else 2)
        seqs_done += 1
    passes = f"{seqs_done / s.batch:.2f} passes over the {s.batch} sequences" if seqs_done > s.batch else \
        f"first {seqs_done} of {s.batch} sequences"
    return {"value": done_bytes / spent / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{passes}, all {s.num_q_heads} query heads, layer 0"
                      f"{' (E4M3 pool)' if fp8 is not None else ''}; {spent:.1f} s of numpy fp64 on one host thread"}


def pack_tensors(tensors, device=None):
    """One contiguous byte buffer (pinned host memory, or device memory) holding
    copies of `tensors` back to back, and views of it with their shapes and
    dtypes.  Offsets stay 16-byte aligned for the sizes used here."""
    sizes = [t.numel() * t.element_size() for t in tensors]
    buf = torch.empty(sum(sizes), dtype=torch.uint8, device=device if device is not None else "cpu")
    if device is None and torch.cuda.is_available():
        buf = buf.pin_memory()
    views, off = [], 0
    for t, n in zip(tensors, sizes):
        v = buf[off:off + n].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
        off += n
    return buf, views


def _oracle_worker(job):
    """One host process of the all-cores baseline: the oracle, as it stands, on
    its share of sequence samples, for about `budget` seconds.  Returns
    (algorithmic bytes covered, seconds spent)."""
    import oracle
    samples, nbytes, budget, scale, dtype, bs, nq, scales = job
    spent, done, i = 0.0, 0.0, 0
    rows = [(0, h) for h in range(nq)]
    while spent < budget:
        k = i % len(samples)
        q, kc, vc, tables, lens = samples[k]
        t0 = time.perf_counter()
        oracle.decode_attention_rows(q, kc, vc, tables, lens, scale, dtype, bs, rows, kv_scales=scales)
        spent += time.perf_counter() - t0
        done += nbytes[k]
        i += 1
    return done, spent


def cpu_baseline_all_cores(w, budget_s: float, fp8=None):
    """The same oracle on every host core: one spawned process per core (BLAS
    held to one thread each), the batch's sequences dealt round-robin, each
    process running for about budget_s seconds.  Throughput = the bytes all
    processes covered over the longest process time."""
    from concurrent.futures import ProcessPoolExecutor
    import multiprocessing as mp
    s = w.spec
    n = max(1, len(os.sched_getaffinity(0)))
    caches = (fp8.k_cache[0], fp8.v_cache[0]) if fp8 is not None else None
    scales = (fp8.k_scale[0].cpu().numpy(), fp8.v_scale[0].cpu().numpy()) if fp8 is not None else None
    kv_elem = 1 if fp8 is not None else 2
    seqs = list(range(min(s.batch, 2 * n)))
    samples = [host_sample(w, [b], caches=caches) for b in seqs]
    nbytes = [row_bytes(w, [w.context_lens[b]] * s.num_q_heads, kv_elem) for b in seqs]
    jobs = []
    for p in range(n):
        mine = list(range(p % len(seqs), len(seqs), n)) or [p % len(seqs)]
        jobs.append(([samples[i] for i in mine], [nbytes[i] for i in mine], budget_s, w.scale, s.dtype, s.block_size,
                     s.num_q_heads, scales))
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    os.environ.update({k: "1" for k in saved})
    try:
        with ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn")) as ex:
            res = list(ex.map(_oracle_worker, jobs))
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    done = sum(r[0] for r in res)
    longest = max(r[1] for r in res)
    return {"value": done / longest / 1e9, "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": f"{n} processes (one per host core, spawn), {len(seqs)} sequences dealt round-robin, all "
                      f"{s.num_q_heads} query heads, layer 0{' (E4M3 pool)' if fp8 is not None else ''}; "
                      f"each about {budget_s:.0f} s of numpy fp64"}


# ----------------------------------------------------------------------------- our arm

def run_ours(args, rank, world, local):
    import paged_kv_cache_26_gb300 as pkv
    from paged_kv_cache_26_gb300 import build as pkv_build
    from paged_kv_cache_26_gb300._native import PkvDims, PkvStepBuffers, lib
    from paged_kv_cache_26_gb300.api import STEP_KEYS

    pkv_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    spec = wl.CONFIGS[args.config]
    if args.batch:
        spec = spec.replace(name=f"{spec.name}_b{args.batch}", batch=args.batch)
    layers = spec.num_layers if args.layers is None else args.layers
    w = wl.generate(spec, seed=args.seed + rank, device=dev, layers=layers)
    s = w.spec
    nl = len(w.q)
    elem = 2
    fp8 = args.kv == "fp8"
    f8 = None
    if fp8:
        if args.splits != 0:
            raise SystemExit("--kv fp8 runs the automatic (persistent) path only: use --splits 0")
        f8 = wl.fp8_caches(w, seed=args.seed + rank)
        w.k_cache, w.v_cache = [], []        # the fp16/bf16 pool is not used
        torch.cuda.empty_cache()
    kv_elem = 1 if fp8 else elem
    L = lib()
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)

    slots_np = pkv.paged_kv_slot_mapping(w.block_tables, w.context_lens, s.block_size)
    slots = torch.from_numpy(slots_np).to(dev)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    outs = [torch.empty_like(q) for q in w.q]
    dims = PkvDims(num_seqs=s.batch, num_q_heads=s.num_q_heads, num_kv_heads=s.num_kv_heads, head_dim=s.head_dim,
                   block_size=s.block_size, num_blocks=w.num_blocks, max_blocks_per_seq=w.max_blocks,
                   dtype=0 if s.dtype == "fp16" else 1)
    splits = int(L.paged_decode_resolve_splits(ctypes.byref(dims), args.splits))
    ws_bytes = int(L.paged_decode_workspace_bytes(ctypes.byref(dims), args.splits))
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    P = ctypes.c_void_p
    scale = ctypes.c_float(w.scale)
    if fp8:
        step_args = [(P(w.q[l].data_ptr()), P(w.k_new[l].data_ptr()), P(w.v_new[l].data_ptr()),
                      P(f8.k_cache[l].data_ptr()), P(f8.v_cache[l].data_ptr()), P(f8.k_scale[l].data_ptr()),
                      P(f8.v_scale[l].data_ptr()), P(bt.data_ptr()), P(cl.data_ptr()), scale,
                      P(outs[l].data_ptr()), P(ws.data_ptr()), ws_bytes, ctypes.byref(dims), sp) for l in range(nl)]
        f_step = L.paged_decode_step_fp8
    else:
        step_args = [(P(w.q[l].data_ptr()), P(w.k_new[l].data_ptr()), P(w.v_new[l].data_ptr()),
                      P(w.k_cache[l].data_ptr()), P(w.v_cache[l].data_ptr()), P(bt.data_ptr()), P(cl.data_ptr()),
                      scale, P(outs[l].data_ptr()), args.splits, P(ws.data_ptr()), ws_bytes, ctypes.byref(dims),
                      sp) for l in range(nl)]
        f_step = L.paged_decode_step

    def step():
        for l in range(nl):
            if f_step(*step_args[l]):
                raise RuntimeError(L.paged_kv_last_error().decode())

    K, W = args.steps, args.warmup
    sampler = ClockSampler(local) if rank == 0 else None
    for _ in range(W):
        step()
    torch.cuda.synchronize()
    pkv.paged_kv_check_status(stream)

    graph = None
    if args.graph:
        # One step (all layers) captured once, replayed each timed step: the
        # library's step allocates nothing, never synchronises and leaves its
        # workspace counters at zero, so a replay is the same step.
        cap = torch.cuda.Stream(dev)
        cap_args = [a[:-1] + (ctypes.c_void_p(cap.cuda_stream),) for a in step_args]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            for l in range(nl):
                if f_step(*cap_args[l]):
                    raise RuntimeError(L.paged_kv_last_error().decode())
        for _ in range(W):
            graph.replay()
        torch.cuda.synchronize()

    # ---- timed region: exactly K steps, no events inside (kernels chain back to back)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    torch.cuda.nvtx.range_push(f"timed {K} steps")
    start.record(stream)
    for _ in range(K):
        if graph is not None:
            graph.replay()
            continue
        for l in range(nl):
            f_step(*step_args[l])
    end.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(world)
    pkv.paged_kv_check_status(stream)
    elapsed_ms = max_over_ranks(start.elapsed_time(end), world, dev)

    # ---- per-launch durations for the roofline: K more steps with an event pair around each call
    n_ev = K * nl
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    i = 0
    for _ in range(K):
        for l in range(nl):
            ev_a[i].record(stream)
            f_step(*step_args[l])
            ev_b[i].record(stream)
            i += 1
    torch.cuda.synchronize()
    clocks = sampler.stop(t_wall0, time.time()) if sampler else None
    pkv.paged_kv_check_status(stream)
    call_ms = [a.elapsed_time(b) for a, b in zip(ev_a, ev_b)]

    attn_b = attention_bytes(w.context_lens, s.batch, s.num_q_heads, s.num_kv_heads, s.head_dim, elem,
                             kv_elem_bytes=kv_elem) * nl
    app_b = append_bytes(s.batch, s.num_kv_heads, s.head_dim, elem, kv_elem_bytes=kv_elem) * nl
    step_bytes = attn_b + app_b
    ms_per_step = elapsed_ms / K
    value = world * step_bytes / (ms_per_step * 1e-3) / 1e9
    peak, peak_kind = load_peaks()
    call_avg_s = statistics.mean(call_ms) * 1e-3
    # The step's launches chain back to back in the K-step region (each may
    # start while the previous one drains); its per-step time is the launch
    # duration the roofline uses.  The isolated per-call time, with an event
    # pair around every call breaking that chaining, is reported beside it.
    step_s = ms_per_step * 1e-3 / nl
    achieved = (step_bytes / nl) / step_s / 1e9
    launches_per_step = 2 if splits == 0 else (2 + (1 if splits > 1 else 0))

    # ---- end to end through the C ABI from pinned host buffers
    # Inputs packed back to back (q, k_new, v_new, tables, lengths) in one pinned
    # host buffer and one device region per layer: one copy in, one copy out.
    host_in = [w.q[0].cpu(), w.k_new[0].cpu(), w.v_new[0].cpu(), torch.from_numpy(w.block_tables),
               torch.from_numpy(w.context_lens)]
    hbuf, hviews = pack_tensors(host_in, device=None)
    keys_in = STEP_KEYS[:-1]
    h = dict(zip(keys_in, hviews))
    h["out"] = torch.empty_like(w.q[0], device="cpu").pin_memory()
    dstage = []
    for l in range(nl):
        dbuf, dviews = pack_tensors(host_in, device=dev)
        dstage.append({**dict(zip(keys_in, dviews)), "out": outs[l], "_buf": dbuf})
    keys = STEP_KEYS
    e2e_args = []
    for l in range(nl):
        bufs = PkvStepBuffers(**{f"{k}_host": h[k].data_ptr() for k in keys},
                              **{f"{k}_dev": dstage[l][k].data_ptr() for k in keys})
        if fp8:
            e2e_args.append((bufs, P(f8.k_cache[l].data_ptr()), P(f8.v_cache[l].data_ptr()),
                             P(f8.k_scale[l].data_ptr()), P(f8.v_scale[l].data_ptr()), scale, P(ws.data_ptr()),
                             ws_bytes, ctypes.byref(dims), sp))
        else:
            e2e_args.append((bufs, P(w.k_cache[l].data_ptr()), P(w.v_cache[l].data_ptr()), scale, args.splits,
                             P(ws.data_ptr()), ws_bytes, ctypes.byref(dims), sp))
    f_e2e = L.paged_decode_step_fp8_from_host if fp8 else L.paged_decode_step_from_host

    def e2e_once():
        for a in e2e_args:
            if f_e2e(ctypes.byref(a[0]), *a[1:]):
                raise RuntimeError(L.paged_kv_last_error().decode())
    for _ in range(min(W, 10)):
        e2e_once()
    torch.cuda.synchronize()
    K_e2e = K
    barrier(world)
    start.record(stream)
    for _ in range(K_e2e):
        e2e_once()
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    pkv.paged_kv_check_status(stream)
    e2e_ms = max_over_ranks(start.elapsed_time(end), world, dev) / K_e2e
    h2d = hbuf.numel() * nl
    d2h = h["out"].numel() * h["out"].element_size() * nl

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3" if fp8 else s.dtype,
        "data": "synthetic (seeded N(0,1) values, scattered block placement"
                + ("; E4M3 pool cast from them with seeded per-head scales)" if fp8 else ")"),
        "config": {"workload": s.name + ("_fp8" if fp8 else ""), "batch": s.batch, "num_q_heads": s.num_q_heads,
                   "num_kv_heads": s.num_kv_heads, "head_dim": s.head_dim, "block_size": s.block_size,
                   "layers_per_step": nl, "context_tokens": int(w.context_lens.sum()),
                   "num_blocks": w.num_blocks,
                   "partition": "persistent, equal blocks per warp" if splits == 0 else f"{splits} splits",
                   "l2": f"no flush: each call streams {attn_b / nl / 2**20:.0f} MiB of K/V, "
                         f"{attn_b / nl / L2_BYTES:.1f}x the 129 MiB L2",
                   "launch": "one CUDA graph per step (captured once, replayed)" if args.graph else
                             "direct C-ABI calls per step",
                   "step": ("paged_decode_step_fp8: E4M3 quantise + append, attention over the E4M3 pool "
                            "(fp16 mma, fp32 softmax), merge" if fp8 else
                            "paged_decode_step: KV append + paged decode attention + merge"),
                   "kv_cache": ("E4M3 codes + f32 per-KV-head K/V scales; q/out " + s.dtype) if fp8 else s.dtype},
        "steps_per_s": round(1e3 / ms_per_step, 2),
        "pct_of_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "roofline": {"bound": "hbm",
                     "kernel": ("paged_decode_step_fp8: decode_persistent_kernel<E4M3> (quantising append fused)"
                                " + merge_persistent_kernel" if fp8 else
                                "paged_decode_step: decode_persistent_kernel (append fused) + merge_persistent_kernel"
                                if splits == 0 else "paged_decode_step: append_at_end_kernel + decode_split_kernel"
                                + (" + merge_split_kernel" if splits > 1 else "")),
                     "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": ncu_traffic(s.name + ("_fp8" if fp8 else "")),
                     "bytes_per_launch": step_bytes // nl, "attention_bytes_per_launch": attn_b // nl,
                     "append_bytes_per_launch": app_b // nl, "avg_launch_us": round(step_s * 1e6, 2),
                     "isolated_call_us": round(call_avg_s * 1e6, 2),
                     "isolated_call_us_p10_p50_p90": [round(float(x) * 1e3, 2)
                                                      for x in np.percentile(call_ms, [10, 50, 90])]},
        "e2e": {"value": round(world * step_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": UNIT,
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": K * nl * launches_per_step,
        "clocks": clocks,
    }
    if s.shared_prefix:
        result["config"]["unique_kv_bytes_per_call"] = unique_kv_bytes(w, kv_elem)
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        one = cpu_baseline(w, args.cpu_budget, fp8=f8)
        try:
            allc = cpu_baseline_all_cores(w, args.cpu_budget, fp8=f8)
            allc["one_thread"] = {"value": one["value"], "cores": 1, "sample": one["sample"]}
            result["cpu_baseline"] = allc
        except Exception as exc:  # the one-thread figure stands alone if processes cannot be started
            one["all_cores_error"] = str(exc)[:200]
            result["cpu_baseline"] = one
    if rank == 0:
        print(json.dumps(result), flush=True)


# ----------------------------------------------------------------------------- several new tokens per sequence

def run_multi(args, rank, world, local):
    """One step = the q_len-token append + multi-token paged decode attention
    (+ split merge) for the whole batch.  Bytes: the one-token formula with q
    and out q_len times larger; the append moves q_len rows per sequence."""
    import oracle
    import paged_kv_cache_26_gb300 as pkv
    from paged_kv_cache_26_gb300 import build as pkv_build
    from paged_kv_cache_26_gb300._native import PkvDims, PkvStepBuffers, lib
    from paged_kv_cache_26_gb300.api import STEP_KEYS

    pkv_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    n = args.q_len
    spec = wl.CONFIGS[args.config]
    if args.batch:
        spec = spec.replace(name=f"{spec.name}_b{args.batch}", batch=args.batch)
    w, m = wl.generate_multi(spec, n, seed=args.seed + rank, device=dev, layers=1)
    s = w.spec
    L = lib()
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    out = torch.empty_like(m.q[0])
    dims = PkvDims(num_seqs=s.batch, num_q_heads=s.num_q_heads, num_kv_heads=s.num_kv_heads, head_dim=s.head_dim,
                   block_size=s.block_size, num_blocks=w.num_blocks, max_blocks_per_seq=w.max_blocks,
                   dtype=0 if s.dtype == "fp16" else 1)
    splits = int(L.paged_decode_multi_resolve_splits(ctypes.byref(dims), n, args.splits))
    ws_bytes = int(L.paged_decode_multi_workspace_bytes(ctypes.byref(dims), n, args.splits))
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    P = ctypes.c_void_p
    step_args = (P(m.q[0].data_ptr()), P(m.k_new[0].data_ptr()), P(m.v_new[0].data_ptr()),
                 P(w.k_cache[0].data_ptr()), P(w.v_cache[0].data_ptr()), P(bt.data_ptr()), P(cl.data_ptr()), n,
                 ctypes.c_float(w.scale), P(out.data_ptr()), args.splits, P(ws.data_ptr()), ws_bytes,
                 ctypes.byref(dims), sp)
    tensor_cores = getattr(args, "tc", False)
    f_step = L.paged_decode_step_multi_tc if tensor_cores else L.paged_decode_step_multi

    def step():
        if f_step(*step_args):
            raise RuntimeError(L.paged_kv_last_error().decode())

    K, W = args.steps, args.warmup
    sampler = ClockSampler(local) if rank == 0 else None
    for _ in range(W):
        step()
    torch.cuda.synchronize()
    pkv.paged_kv_check_status(stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start.record(stream)
    for _ in range(K):
        f_step(*step_args)
    end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop(t_wall0, time.time()) if sampler else None
    barrier(world)
    pkv.paged_kv_check_status(stream)
    ms_per_step = max_over_ranks(start.elapsed_time(end), world, dev) / K

    elem = 2
    kv_b = attention_bytes(w.context_lens, s.batch, s.num_q_heads, s.num_kv_heads, s.head_dim, elem)
    kv_b += 2 * s.batch * (n - 1) * s.num_q_heads * s.head_dim * elem          # q and out of the extra tokens
    app_b = append_bytes(s.batch * n, s.num_kv_heads, s.head_dim, elem)
    step_bytes = kv_b + app_b
    value = world * step_bytes / (ms_per_step * 1e-3) / 1e9
    peak, peak_kind = load_peaks()

    # ---- end to end through the C ABI from pinned host buffers: inputs packed back
    # to back in one pinned buffer and one device region (one copy in, one out)
    host_in = [m.q[0].cpu(), m.k_new[0].cpu(), m.v_new[0].cpu(), torch.from_numpy(w.block_tables),
               torch.from_numpy(w.context_lens)]
    hbuf, hviews = pack_tensors(host_in, device=None)
    dbuf, dviews = pack_tensors(host_in, device=dev)
    keys_in = STEP_KEYS[:-1]
    h = dict(zip(keys_in, hviews))
    h["out"] = torch.empty_like(out, device="cpu").pin_memory()
    dst = {**dict(zip(keys_in, dviews)), "out": out}
    bufs = PkvStepBuffers(**{f"{k}_host": h[k].data_ptr() for k in STEP_KEYS},
                          **{f"{k}_dev": dst[k].data_ptr() for k in STEP_KEYS})
    f_e2e = L.paged_decode_step_multi_from_host
    e2e_args = (ctypes.byref(bufs), n, P(w.k_cache[0].data_ptr()), P(w.v_cache[0].data_ptr()),
                ctypes.c_float(w.scale), args.splits, P(ws.data_ptr()), ws_bytes, ctypes.byref(dims), sp)

    def e2e_once():
        if f_e2e(*e2e_args):
            raise RuntimeError(L.paged_kv_last_error().decode())

    for _ in range(min(W, 10)):
        e2e_once()
    torch.cuda.synchronize()
    barrier(world)
    start.record(stream)
    for _ in range(K):
        e2e_once()
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(start.elapsed_time(end), world, dev) / K
    h2d = hbuf.numel()
    d2h = h["out"].numel() * h["out"].element_size()

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": s.dtype, "data": "synthetic (seeded N(0,1) values, scattered block placement)",
        "config": {"workload": f"{s.name}_q{n}", "batch": s.batch, "q_len": n, "num_q_heads": s.num_q_heads,
                   "num_kv_heads": s.num_kv_heads, "head_dim": s.head_dim, "block_size": s.block_size,
                   "context_tokens": int(w.context_lens.sum()), "num_blocks": w.num_blocks,
                   "partition": f"{splits} splits per sequence",
                   "l2": f"no flush: each call streams {kv_b / 2**20:.0f} MiB, {kv_b / L2_BYTES:.1f}x the 129 MiB L2",
                   "step": ("paged_decode_step_multi_tc" if tensor_cores else "paged_decode_step_multi")
                           + ": q_len-token KV append + causal multi-token paged attention"
                           + (" + merge" if splits > 1 else ""),
                   **({"e2e_step": "paged_decode_step_multi_from_host (the default kernel: there is no "
                                   "host-buffer tcgen05 step)"} if tensor_cores else {})},
        "steps_per_s": round(1e3 / ms_per_step, 2),
        "query_tokens_per_s": round(world * s.batch * n * 1e3 / ms_per_step, 1),
        "roofline": {"bound": "hbm", "kernel": "paged_decode_step_multi: append_multi_kernel + "
                     + ("decode_multi_tc_kernel (tcgen05)" if tensor_cores
                        else "decode_multi_rows_kernel" if s.num_q_heads // s.num_kv_heads * n > 8
                        else "decode_multi_query_kernel") + (" + merge_split_kernel" if splits > 1 else ""),
                     "achieved": round(step_bytes / (ms_per_step * 1e-3) / 1e9, 1), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(step_bytes / (ms_per_step * 1e-3) / 1e9 / peak, 4), "traffic": None,
                     "bytes_per_launch": step_bytes, "avg_launch_us": round(ms_per_step * 1e3, 2)},
        "e2e": {"value": round(world * step_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": UNIT,
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": K * (3 if splits > 1 else 2),
        "clocks": clocks,
    }
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        # the oracle over the batch's sequences in order (all tokens and heads) for about cpu_budget seconds
        qb = m.q[0].cpu().view(torch.int16).numpy().view(np.uint16)
        spent, done, nseq = 0.0, 0.0, 0
        while spent < args.cpu_budget:
            b = nseq % s.batch
            sample = host_sample(w, [b])
            rows = [(0, i, hh) for i in range(n) for hh in range(s.num_q_heads)]
            t0 = time.perf_counter()
            oracle.decode_attention_multi(qb[[b]], sample[1], sample[2], sample[3], sample[4], n, w.scale, s.dtype,
                                          s.block_size, rows=rows)
            spent += time.perf_counter() - t0
            done += row_bytes(w, [w.context_lens[b]] * s.num_q_heads) + 2 * (n - 1) * s.num_q_heads * s.head_dim * 2
            nseq += 1
        result["cpu_baseline"] = {"value": done / spent / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
                                  "sample": f"{nseq} sequences in order, all {n} tokens x {s.num_q_heads} heads; "
                                            f"{spent:.1f} s of numpy fp64 on one host thread (the cache as left "
                                            f"by the timed steps)"}
    if rank == 0:
        print(json.dumps(result), flush=True)


# ----------------------------------------------------------------------------- copy-on-write

def run_cow(args, rank, world, local):
    """Copy-on-write block copies at this configuration's block shape: one
    step = paged_kv_copy_blocks of `--cow-pairs` random (src, dst) block pairs
    of the K and V pools.  Bytes: each pair reads and writes one block of K and
    one of V."""
    import oracle
    import paged_kv_cache_26_gb300 as pkv
    from paged_kv_cache_26_gb300 import build as pkv_build

    pkv_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    spec = wl.CONFIGS[args.config]
    n = args.cow_pairs
    nb = max(4 * n, 1024)
    dt = wl.DTYPES[spec.dtype]
    g = torch.Generator(device=dev)
    g.manual_seed(args.seed + rank)
    kc = torch.randn((nb, spec.num_kv_heads, spec.block_size, spec.head_dim), generator=g, device=dev).to(dt)
    vc = torch.randn_like(kc)
    perm = np.random.default_rng(args.seed + rank).permutation(nb)
    pairs_np = np.stack([perm[:n], perm[n:2 * n]], 1).astype(np.int32)
    pairs = torch.from_numpy(pairs_np).to(dev)
    block_bytes = spec.num_kv_heads * spec.block_size * spec.head_dim * kc.element_size()
    step_bytes = 2 * 2 * block_bytes * n
    stream = torch.cuda.current_stream(dev)
    K, W = args.steps, args.warmup
    for _ in range(W):
        pkv.paged_kv_copy_blocks(kc, vc, pairs)
    torch.cuda.synchronize()
    pkv.paged_kv_check_status(stream)
    sampler = ClockSampler(local) if rank == 0 else None
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start.record(stream)
    for _ in range(K):
        pkv.paged_kv_copy_blocks(kc, vc, pairs)
    end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop(t_wall0, time.time()) if sampler else None
    barrier(world)
    pkv.paged_kv_check_status(stream)
    ms = max_over_ranks(start.elapsed_time(end), world, dev) / K
    peak, peak_kind = load_peaks()
    achieved = step_bytes / (ms * 1e-3) / 1e9
    # end to end: the pair list copied in from pinned host memory each step, a word read back
    hp = torch.from_numpy(pairs_np).pin_memory()
    flag = torch.empty(1, dtype=torch.int32).pin_memory()
    barrier(world)
    start.record(stream)
    for _ in range(K):
        pairs.copy_(hp, non_blocking=True)
        pkv.paged_kv_copy_blocks(kc, vc, pairs)
        flag.copy_(pairs[0, :1], non_blocking=True)
    end.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(start.elapsed_time(end), world, dev) / K
    result = {
        "metric": METRIC, "value": round(world * achieved, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": spec.dtype, "data": "synthetic (seeded N(0,1) blocks, seeded pairs)",
        "config": {"workload": f"{spec.name}_cow{n}", "pairs": n, "num_blocks": nb,
                   "block_bytes_per_cache": block_bytes,
                   "l2": f"no flush: each call moves {step_bytes / 2**20:.0f} MiB over a "
                         f"{2 * nb * block_bytes / 2**20:.0f} MiB pool",
                   "step": "paged_kv_copy_blocks: copy-on-write of n shared blocks (K and V)"},
        "roofline": {"bound": "hbm", "kernel": "copy_blocks_kernel", "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": None,
                     "bytes_per_launch": step_bytes, "avg_launch_us": round(ms * 1e3, 2)},
        "e2e": {"value": round(world * step_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": UNIT,
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": int(pairs_np.nbytes), "d2h_bytes_per_step": 4},
        "gpu_launches": K,
        "clocks": clocks,
    }
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        # the oracle works on a host copy of the touched blocks
        idx = torch.from_numpy(np.unique(pairs_np)).to(dev)
        remap = {int(b): i for i, b in enumerate(np.unique(pairs_np))}
        hk = kc.index_select(0, idx).cpu().view(torch.int16).numpy()
        hv = vc.index_select(0, idx).cpu().view(torch.int16).numpy()
        local_pairs = [(remap[int(a)], remap[int(b)]) for a, b in pairs_np]
        spent, calls = 0.0, 0
        while spent < args.cpu_budget:
            t0 = time.perf_counter()
            oracle.copy_blocks(hk, hv, local_pairs)
            spent += time.perf_counter() - t0
            calls += 1
        result["cpu_baseline"] = {"value": calls * step_bytes / spent / 1e9, "unit": UNIT, "cores": 1,
                                  "kind": "oracle", "sample": f"{calls} full calls ({n} pairs each) on a host copy "
                                                              f"of the touched blocks, {spent:.1f} s, one thread"}
    if rank == 0:
        print(json.dumps(result), flush=True)


# ----------------------------------------------------------------------------- continuous batching

def run_loop(args, rank, world, local):
    """Continuous batching at this configuration's shape: args.batch (or the
    configuration's batch) slots; prompts drawn from its length law, 32..256
    generated tokens each; finished sequences leave and waiting ones are
    admitted every step.  Reports steps/s, generated tokens/s, attention GB/s
    and the allocator's unused tail per sequence."""
    from paged_kv_cache_26_gb300 import build as pkv_build
    from paged_kv_cache_26_gb300.loop import DecodeLoop
    import paged_kv_cache_26_gb300 as pkv

    pkv_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    spec = wl.CONFIGS[args.config]
    B = args.batch or spec.batch
    dt = wl.DTYPES[spec.dtype]
    rng = np.random.default_rng(args.seed + rank)
    max_prompt = int(wl.draw_lengths(spec.replace(batch=4096), np.random.default_rng(1)).max())
    max_ctx = max_prompt + 256
    num_blocks = int(math.ceil(1.25 * B * max_ctx / 16))
    fp8 = args.kv == "fp8"
    scales = {}
    if fp8:
        # Seeded per-KV-head scales of the E4M3 pool, as the fixed-batch workloads draw them.
        srng = np.random.default_rng(args.seed + rank + 7)
        scales = {n: torch.tensor(srng.uniform(0.004, 0.02, size=spec.num_kv_heads), dtype=torch.float32,
                                  device=dev) for n in ("k_scale", "v_scale")}
    loop = DecodeLoop(num_blocks, spec.num_q_heads, spec.num_kv_heads, spec.head_dim, B, max_ctx, dt, dev,
                      args.seed + rank, **scales)
    g = torch.Generator(device=dev).manual_seed(args.seed + rank)
    prompt_k = torch.randn(max_prompt, spec.num_kv_heads, spec.head_dim, generator=g, device=dev).to(dt)
    prompt_v = torch.randn_like(prompt_k)
    q = torch.randn(B, spec.num_q_heads, spec.head_dim, generator=g, device=dev).to(dt)
    kn = torch.randn(B, spec.num_kv_heads, spec.head_dim, generator=g, device=dev).to(dt)
    vn = torch.randn_like(kn)
    # The arrival queue: prompt lengths from the configuration's length law,
    # 32..256 generated tokens each, drawn up front (requests wait in it).
    n_queue = B + (args.steps + args.warmup) * B // 16 + 64
    queue_p = wl.draw_lengths(spec.replace(batch=n_queue), rng).astype(np.int64)
    queue_g = rng.integers(32, 257, size=n_queue)
    counts = {"admitted": 0, "retired": 0, "next": 0}

    def admit_all():
        while loop.num_free_slots:
            i = counts["next"] % n_queue
            P = int(queue_p[i])
            if loop.admit(prompt_k[:P], prompt_v[:P], int(queue_g[i])) is None:
                break
            counts["next"] += 1
            counts["admitted"] += 1

    def one_step():
        admit_all()
        loop.step(q, kn, vn)
        counts["retired"] += len(loop.finish_step())

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    counts.update(admitted=0, retired=0)
    loop.reset_stats()
    barrier(world)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    start.record()
    for _ in range(args.steps):
        one_step()
    end.record()
    torch.cuda.synchronize()
    wall_s = time.perf_counter() - t0
    pkv.paged_kv_check_status()
    gpu_s = max_over_ranks(start.elapsed_time(end) * 1e-3, world, dev)
    wall_s = max_over_ranks(wall_s, world, dev)
    st = loop.stats()
    elem, kv_elem = 2, (1 if fp8 else 2)
    blocks = (st["context_tokens"] + st["unused_tail_slots"]) // 16
    kv_bytes = (st["context_tokens"] * spec.num_kv_heads * spec.head_dim * 2 * kv_elem
                + st["steps"] * (2 * B * spec.num_q_heads * spec.head_dim * elem + 4 * B) + 4 * blocks)
    tokens = st["sequence_steps"]
    if rank == 0:
        print(json.dumps({
            "metric": "continuous-batching decode steps/s (paged_decode_step per step, host scheduling included)",
            "value": round(world * args.steps / wall_s, 2), "unit": "steps/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(wall_s / args.steps * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "dtype": "e4m3" if fp8 else spec.dtype, "data": "synthetic",
            "config": {"workload": f"{spec.name} continuous batching" + (", E4M3 pool" if fp8 else ""),
                       "batch_slots": B,
                       "prompt_lengths": str(spec.lengths), "generated_tokens": "U[32,256]",
                       "num_blocks": num_blocks},
            "generated_tokens_per_s": round(world * tokens / wall_s, 1),
            "attention_GBs": round(world * kv_bytes / wall_s / 1e9, 1),
            "gpu_busy_frac": round(gpu_s / wall_s, 3),
            "mean_unused_tail_blocks": round(st["unused_tail_slots"] / max(1, st["sequence_steps"]) / 16, 3),
            "admitted": counts["admitted"], "retired": counts["retired"],
        }), flush=True)


# ----------------------------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    """The fp64 oracle on the host cores, on this arm's workload.  Each step is
    a bounded sample of (sequence, query head) rows, sized so that the whole
    run stays within about args.ref_budget seconds."""
    if rank != 0:
        return
    spec = wl.CONFIGS[args.config]
    device = "cuda" if torch.cuda.is_available() else "cpu"
    w = wl.generate(spec, seed=args.seed, device=device, layers=1)
    s = w.spec
    rng = np.random.default_rng(args.seed)
    seqs = sorted(rng.choice(s.batch, size=min(4, s.batch), replace=False).tolist())
    sample = host_sample(w, seqs)
    all_rows = [(i, h) for i in range(len(seqs)) for h in range(s.num_q_heads)]
    t_row = oracle_rows_timed(w, sample, all_rows[:4]) / 4
    per_step = args.ref_budget / max(1, args.steps + args.warmup)
    n_rows = int(min(len(all_rows), max(1, per_step / max(t_row, 1e-6))))
    rows = all_rows[:n_rows]
    lens_rows = [int(sample[4][i]) for i, _ in rows]
    for _ in range(args.warmup):
        oracle_rows_timed(w, sample, rows)
    spent = sum(oracle_rows_timed(w, sample, rows) for _ in range(args.steps))
    step_s = spent / args.steps
    value = row_bytes(w, lens_rows) / step_s / 1e9
    desc = (f"{n_rows} (sequence, query head) rows of sequences {seqs} per step, layer 0; "
            f"numpy fp64 on one host thread")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) values, scattered block placement)",
        "config": {"workload": s.name, "batch": s.batch, "num_q_heads": s.num_q_heads,
                   "num_kv_heads": s.num_kv_heads, "head_dim": s.head_dim, "block_size": s.block_size},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="llama3_8b_b64", choices=sorted(wl.CONFIGS))
    ap.add_argument("--splits", type=int, default=0, help="0 = automatic, 1 = single pass, n = n splits")
    ap.add_argument("--layers", type=int, default=None, help="cap on layer caches (multi-layer configs)")
    ap.add_argument("--batch", type=int, default=None, help="override the configuration's batch size")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=60.0, help="seconds of oracle work for --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kv", choices=["native", "fp8"], default="native",
                    help="pool format: the configuration's fp16/bf16, or E4M3 codes with per-head scales")
    ap.add_argument("--loop", action="store_true", help="continuous-batching loop instead of the fixed batch")
    ap.add_argument("--q-len", type=int, default=1, help="new tokens per sequence (>1: multi-token decode)")
    ap.add_argument("--tc", action="store_true",
                    help="multi-token decode on the tcgen05 kernel (64 query rows per KV head; the e2e leg keeps "
                         "the default host-buffer step)")
    ap.add_argument("--cow", action="store_true", help="copy-on-write block copies instead of the decode step")
    ap.add_argument("--graph", action="store_true", help="capture the step in a CUDA graph and replay it")
    ap.add_argument("--cow-pairs", type=int, default=2048, help="block pairs per copy-on-write call")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.loop:
        run_loop(args, rank, world, local)
    elif args.q_len > 1:
        run_multi(args, rank, world, local)
    elif args.cow:
        run_cow(args, rank, world, local)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

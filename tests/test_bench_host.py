"""Host-side checks of bench.py: its bytes model against the oracle's
accounting, the multi-rank timing helpers on two gloo ranks (CPU), the
reference arm's rank handling, and the stale-profile rule for ncu traffic."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle


def test_attention_bytes_match_the_oracle_accounting():
    rng = np.random.default_rng(0)
    for _ in range(50):
        B = int(rng.integers(1, 40))
        lens = rng.integers(0, 5000, size=B)
        hkv = int(rng.choice([1, 2, 8, 32]))
        g = int(rng.choice([1, 4, 8]))
        d = int(rng.choice([64, 128]))
        entries = int(((lens + 15) // 16).sum())
        assert bench.attention_bytes(lens, B, hkv * g, hkv, d, 2) == \
            oracle.attention_call_bytes(lens, B, hkv * g, hkv, d, 2, entries)


def test_append_bytes():
    # read + write of the new K and V rows, plus the slot mapping
    assert bench.append_bytes(64, 8, 128, 2) == 2 * (2 * 64 * 8 * 128 * 2) + 4 * 64


def test_llama3_8b_bytes_per_call_matches_the_stated_figure():
    # Llama-3-8B-shaped batch: ~2304 tokens mean x 64 sequences x 4096 B per
    # token (8 KV heads x 128 x 2 x 2 B) is about 604 MB of K/V per call.
    import workloads as wl
    w = wl.generate(wl.LLAMA3_8B.replace(batch=64), seed=0, layers=0)
    b = bench.attention_bytes(w.context_lens, 64, 32, 8, 128, 2)
    assert 0.5e9 < b < 0.7e9


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    r, w, _ = bench.dist_setup()
    assert (r, w) == (rank, world)
    bench.barrier(world)
    slowest = bench.max_over_ranks(10.0 + rank, world, torch.device("cpu"))
    q.put((rank, slowest))
    dist.destroy_process_group()


def test_max_over_ranks_on_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 11.0), (1, 11.0)]


def test_reference_arm_runs_on_rank_zero_only(capsys):
    import types
    args = types.SimpleNamespace(config="tiny", seed=0, steps=3, warmup=3, ref_budget=1.0)
    bench.run_reference(args, rank=1, world=2)
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_one_line_on_cpu(capsys):
    import json
    import types
    args = types.SimpleNamespace(config="tiny", seed=0, steps=3, warmup=3, ref_budget=1.0)
    bench.run_reference(args, rank=0, world=1)
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_ncu_traffic_is_dropped_when_the_kernel_changed(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "profiles").mkdir()
    csrc = tmp_path / "paged_kv_cache_26_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in bench.DECODE_KERNEL_SOURCES:
        (csrc / name).write_text("one")
    h = bench.kernel_source_hash()
    (tmp_path / "profiles" / "decode_persistent_kernel_x.md").write_text(
        f"source_sha256: {h}\ntraffic_bytes_per_launch: 123\n")
    assert bench.ncu_traffic("x") == 123.0
    (csrc / "other_kernel.cuh").write_text("a kernel the profile does not describe")
    assert bench.ncu_traffic("x") == 123.0
    (csrc / bench.DECODE_KERNEL_SOURCES[0]).write_text("two")
    assert bench.ncu_traffic("x") is None


def test_repository_python_compiles_without_warnings():
    # A warning at compile time (for example a string literal followed by a
    # parenthesised expression, which Python reads as a call) is a bug that
    # only shows when that line runs.
    import glob
    import warnings
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    files = [os.path.join(root, f) for f in ("bench.py", "__graft_entry__.py")]
    for d in ("paged_kv_cache_26_gb300", "oracle", "workloads", "tests"):
        files += glob.glob(os.path.join(root, d, "**", "*.py"), recursive=True)
    for f in files:
        with open(f) as fh:
            src = fh.read()
        with warnings.catch_warnings():
            warnings.simplefilter("error")
            compile(src, f, "exec")


@pytest.mark.parametrize("q_len", [1, 4, 8])
def test_shared_prefix_sequences_never_append_into_the_shared_blocks(q_len):
    # Sequences that share the prefix blocks must write their new tokens into
    # blocks of their own (an engine copies a shared block before writing it).
    import workloads as wl
    w, _ = wl.generate_multi(wl.LLAMA70B_TAIL.replace(batch=256), q_len, seed=0, layers=1)
    prefix_blocks = wl.LLAMA70B_TAIL.shared_prefix[1] // wl.LLAMA70B_TAIL.block_size
    shared = set(int(x) for x in w.block_tables[w.shared_seqs[0], :prefix_blocks])
    for b in range(w.spec.batch):
        L = int(w.context_lens[b])
        for pos in range(max(0, L - q_len), L):
            assert int(w.block_tables[b, pos // w.spec.block_size]) not in shared or b not in w.shared_seqs

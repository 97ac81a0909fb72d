"""CPU checks of bench.py: multi-rank aggregation (world size 2 over gloo),
the algorithmic byte count, and the reference (oracle) arm's JSON line."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
import workloads  # noqa: E402


def _rank_main(rank, world, port, ms_by_rank, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mx = bench.max_over_ranks(ms_by_rank[rank], world)
        val = bench.aggregate_value(1_000_000_000, world, mx)
        out_q.put((rank, mx, val))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    ms = [0.25, 0.5]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, val in res:
        assert mx == 0.5                      # every rank sees the slowest rank's time
        assert val == pytest.approx(2 * 1e9 / 0.5e-3 / 1e9)


def test_single_rank_passthrough():
    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.aggregate_value(2_000_000_000, 1, 1.0) == pytest.approx(2000.0)


def test_algorithmic_bytes_decode_gqa():
    wl = workloads.decode_gqa()
    ab = bench.algorithmic_bytes(wl)
    n = wl.total_lens
    assert ab["kv"] == int(n.sum()) * 2 * 8 * 128 * 2
    assert ab["q"] == 64 * 32 * 128 * 2 and ab["out"] == 64 * 32 * 128 * 4
    assert ab["tables"] == int(np.ceil(n / 16).sum()) * 4
    assert ab["decode_total"] == ab["kv"] + ab["q"] + ab["out"] + ab["tables"] + ab["lens"]
    assert 5.0e8 < ab["kv"] < 6.2e8       # about 554 MB of K/V per step


def test_algorithmic_bytes_with_a_window():
    wl = workloads.decode_gqa()
    full = bench.algorithmic_bytes(wl)
    # a window at least as long as every context moves exactly the full bytes
    assert bench.algorithmic_bytes(wl, int(wl.total_lens.max())) == full
    w = 100
    ab = bench.algorithmic_bytes(wl, w)
    n = wl.total_lens.astype(np.int64)
    vis = np.minimum(n, w)
    assert ab["kv"] == int(vis.sum()) * 2 * 8 * 128 * 2
    # pages from the one holding position n - w to the one holding n - 1
    lo = np.maximum(n - w, 0)
    pages = (n - 1) // 16 - lo // 16 + 1
    assert ab["tables"] == int(pages.sum()) * 4
    assert ab["q"] == full["q"] and ab["out"] == full["out"]


def _distinct_rows(wl, tables, window=0):
    # set of (physical block, offset) pairs any sequence reads
    seen = set()
    for s, table in enumerate(tables):
        n = int(wl.total_lens[s])
        lo = max(n - window, 0) if window else 0
        seen |= {(table[i // wl.block_size], i % wl.block_size) for i in range(lo, n)}
    return len(seen)


def test_physical_bytes_equal_logical_without_sharing():
    import oracle
    wl = workloads.decode_gqa(scale=1 / 16)
    tables = oracle.OracleCache(wl).tables
    assert bench.physical_kv_bytes(wl, tables) == bench.algorithmic_bytes(wl)["kv"]
    assert bench.physical_kv_bytes(wl, tables, 50) == bench.algorithmic_bytes(wl, 50)["kv"]


def test_physical_bytes_count_a_shared_prefix_once():
    import oracle
    wl = workloads.decode_long_shared(scale=1 / 256)
    tables = oracle.OracleCache(wl).tables
    per_token = 2 * wl.num_kv_heads * wl.head_dim * 2
    phys = bench.physical_kv_bytes(wl, tables)
    assert phys == _distinct_rows(wl, tables) * per_token
    # logical - physical = the rows of every pair's fully shared pages (the
    # partly filled shared page is copied on write, so it is not shared)
    shared = 0
    for s in range(wl.num_seqs):
        p = int(wl.pair_of[s])
        if p > s:
            shared += int(wl.prefix_len[s]) // wl.block_size * wl.block_size
    assert shared > 0
    assert bench.algorithmic_bytes(wl)["kv"] - phys == shared * per_token
    w = 200
    assert bench.physical_kv_bytes(wl, tables, w) == _distinct_rows(wl, tables, w) * per_token


def test_prefill_flops_matches_closed_form():
    wl = workloads.prefill()
    # 16 sequences, queries at positions 2048..2559 see pos+1 keys
    vis = 16 * sum(2048 + 1 + i for i in range(512))
    assert bench.prefill_flops(wl) == 4.0 * 128 * 32 * vis
    assert abs(bench.prefill_flops(wl) / 1e9 - 309.3) < 0.1


def test_reference_arm_prints_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "decode_tiny", "--steps", "3", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for k in ("metric", "value", "unit", "cpu_baseline", "e2e", "config"):
        assert k in line
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_runs_on_rank_0_only():
    # under torchrun every rank but 0 exits at once, printing nothing
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--workload", "decode_tiny", "--steps", "3", "--warmup",
                        "1"], capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_recorded_traffic_is_dropped_when_the_sources_change(monkeypatch):
    import json as _json
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        records = _json.load(f)
    kernel = sorted(records)[0]
    workload = sorted(records[kernel])[0]
    rec = records[kernel][workload]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: rec["source_hash"])
    assert bench.recorded_traffic(kernel, workload) == rec["dram_bytes_per_launch"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: "0" * 16)
    assert bench.recorded_traffic(kernel, workload) is None
    assert bench.recorded_traffic(kernel, "no_such_workload") is None


def test_recorded_traffic_is_one_launch_of_read_plus_write():
    import json as _json
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        records = _json.load(f)
    for kernel, by_workload in records.items():
        assert kernel in bench.KERNEL_SOURCES, kernel
        for workload, rec in by_workload.items():
            captured = rec["dram_read"] + rec["dram_write"]
            if rec.get("captured_scale", 1.0) == 1.0:
                assert rec["dram_bytes_per_launch"] == captured, (kernel, workload)
            else:  # a smaller case scaled to the full workload by its bytes
                assert rec["dram_bytes_per_launch"] > captured, (kernel, workload)


def test_kernel_source_hash_covers_device_code_only():
    h = bench.kernel_source_hash("decode_mma_kernel")
    assert len(h) == 16 and h == bench.kernel_source_hash("decode_mma_kernel")
    assert h != bench.kernel_source_hash("decode_partition_kernel")

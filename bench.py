#!/usr/bin/env python
"""Benchmark of the paged KV-cache attention hot path; prints ONE JSON line.

A decode step is one pass of the decode hot path over one batch: pa_write_kv
of the batch's new K/V rows through slot_mapping, then pa_decode (split-KV
partition kernel + merge kernel) reading every visible token through the
block tables.  A prefill step is pa_write_kv + pa_prefill.

Default (``--workload suite``): the line's top level is the headline
configuration, the MHA decode batch (256 sequences, 32/32 heads, head_dim
128, block size 16, bf16, contexts lognormal(ln 512, 1) clipped to [16,
2048]; the largest single-GPU decode batch, 2.86 GB of K/V per step).
``suite`` holds one record per other configuration (the tiny fp32 decode,
the GQA decode, the long shared-prefix decode also through
pa_decode_shared and with FP8 pages, the chunked prefill) and the pa_write_kv / pa_copy_blocks
microbenchmarks, each with its own value, kernel times, roofline and clocks.
``--workload NAME`` times one workload only.

Timing: W untimed warm-up steps; then K steps bracketed by CUDA events on the
launching stream; barrier + synchronize around the loop; max over ranks.
Steps that move less than twice the 129 MB L2 (and ``--l2 flush``) get a
256 MiB write before every step, then a read of the same buffer (so the
write's dirty lines are written back before the step), both outside its
events.  ``--path fused`` times
pa_decode_step (one launch) and ``--window W`` pa_decode_window instead.
value = algorithmic bytes of all ranks / max step time (GB/s).  The
algorithmic bytes of a decode step are the K/V rows of every visible token,
Q, the fp32 output, the block-table entries and context lengths.

--impl reference times the float64 CPU oracle on the host cores instead (the
only other code this script may run from oracle/).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "paged decode KV-read GB/s (% of HBM peak) and decode tokens/s on 1 GB300"
L2_FLUSH_BYTES = 256 << 20


def flush_l2(buf, i: int):
    """Write a buffer twice the size of L2 (so L2 holds none of the step's
    data), then read it back so the lines the write left dirty are written
    back now rather than inside the next timed kernel."""
    import torch
    buf.fill_(i & 255)
    buf.view(torch.int64).sum()  # int64: the sum needs no widened copy of the buffer


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="suite", choices=["suite"] + sorted(workloads.WORKLOADS),
                    help="suite (default): the headline decode_mha line with a record per other "
                         "configuration and the write / copy microbenchmarks; or one workload")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--l2", choices=["none", "flush"], default="none",
                    help="none: the step's K/V (4x the 129 MB L2) is itself larger than L2; "
                         "flush: write a 256 MiB buffer before every timed step")
    ap.add_argument("--scale", type=float, default=1.0,
                    help="single-workload runs: the workload's size scale (small profiling cases)")
    ap.add_argument("--path", choices=["fused", "split", "shared"], default="split",
                    help="decode step: split = pa_write_kv + pa_decode_partial + pa_decode_merge "
                         "(dependent launches; fastest on large batches); fused = pa_decode_step "
                         "(write + attention + merge in one launch; fastest on small batches); "
                         "shared = pa_write_kv + pa_decode_shared (declared shared-prefix pairs)")
    ap.add_argument("--window", type=int, default=0,
                    help="decode: sliding window in positions (pa_decode_window); 0 = none")
    ap.add_argument("--partition-tokens", type=int, default=0,
                    help="split-KV partition size for decode (0 = the library's choice)")
    return ap.parse_args()


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def algorithmic_bytes(wl, window: int = 0) -> dict:
    """Bytes one decode (or prefill) step must move at minimum (with a sliding
    window: only the last `window` positions and the pages holding them)."""
    e = wl.elem_bytes
    n = wl.total_lens.astype(np.int64)
    lo = np.maximum(n - window, 0) if window > 0 else np.zeros_like(n)
    kv = int((n - lo).sum()) * wl.logical_bytes_per_token()
    tables = int((-(-n // wl.block_size) - lo // wl.block_size).sum()) * 4
    n_q = int(wl.new_lens.sum())
    q = n_q * wl.num_q_heads * wl.head_dim * e
    out = n_q * wl.num_q_heads * wl.head_dim * 4
    lens = wl.num_seqs * 4
    write = n_q * wl.num_kv_heads * wl.head_dim * e * 2 * 2 + n_q * 8
    return {"kv": kv, "q": q, "out": out, "tables": tables, "lens": lens, "write": write,
            "decode_total": kv + q + out + tables + lens}


def physical_kv_bytes(wl, tables, window: int = 0) -> int:
    """K/V bytes of the distinct physical pages one decode step reads.  A page
    that several sequences reference (a forked prefix) counts once, with the
    union of the rows they read from it; the logical count in
    algorithmic_bytes counts it once per sequence."""
    bp = wl.block_size
    rows = {}
    for s, table in enumerate(tables):
        n = int(wl.total_lens[s])
        lo = max(n - window, 0) if window > 0 else 0
        for j in range(lo // bp, -(-n // bp)):
            a, b = max(j * bp, lo) - j * bp, min((j + 1) * bp, n) - j * bp
            blk = int(table[j])
            rows[blk] = rows.get(blk, 0) | (((1 << (b - a)) - 1) << a)
    return sum(bin(m).count("1") for m in rows.values()) * wl.logical_bytes_per_token()


def ab_kv_mb(wl, window: int = 0) -> float:
    return algorithmic_bytes(wl, window)["kv"] / 1e6


def prefill_flops(wl) -> float:
    """Causal-visible flops of one prefill pass: 4*D per (query, head, visible key)."""
    tot = 0
    for s in range(wl.num_seqs):
        c, m = int(wl.cached_lens[s]), int(wl.new_lens[s])
        vis = (c + 1 + np.arange(m)) if wl.causal else np.full(m, c + m)
        tot += int(vis.sum())
    return 4.0 * wl.head_dim * wl.num_q_heads * tot


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) while the timed loop runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        time.sleep(0.15)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- traffic record
# The source text each kernel's device code comes from.  decode.cu is taken
# only up to the include of the tensor-core headers: everything after it is
# the merge kernel and host code (plans, dispatch), which do not change what a
# partition kernel reads or writes.
_DECODE_DEVICE = ("decode.cu", '#include "decode_mma.cuh"')
KERNEL_SOURCES = {
    "decode_partition_kernel": (_DECODE_DEVICE, "common.cuh"),
    "decode_step": (_DECODE_DEVICE, "decode_mma.cuh", "tcgen05.cuh", "common.cuh"),
    "decode_mma_kernel": (_DECODE_DEVICE, "decode_mma.cuh", "tcgen05.cuh", "common.cuh"),
    "decode_shared_kernel": (_DECODE_DEVICE, "decode_mma.cuh", "tcgen05.cuh", "common.cuh"),
    "decode_fp8_mma_kernel": (_DECODE_DEVICE, "decode_mma_fp8.cuh", "tcgen05.cuh", "common.cuh"),
    "prefill_kernel": ("prefill.cu", "tcgen05.cuh", "common.cuh"),
}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the source text a kernel's device code comes from (to tell
    whether a recorded ncu traffic figure still describes the kernel)."""
    h = hashlib.sha256()
    for src in KERNEL_SOURCES[kernel]:
        name, stop = (src, None) if isinstance(src, str) else src
        with open(os.path.join(ROOT, "paged_kv_cache_148_gb300", "csrc", name), "rb") as fh:
            text = fh.read()
        if stop is not None:
            cut = text.find(stop.encode())
            if cut < 0:
                raise ValueError("%s: marker %r not found" % (name, stop))
            text = text[:cut]
        h.update(text)
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        rec = d[kernel][workload]
        if rec.get("source_hash") == kernel_source_hash(kernel):
            return int(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# --------------------------------------------------------------------------- CPU oracle
def cpu_oracle_run(wl, seconds: float):
    """Time the float64 oracle on the host cores over a bounded sample of the batch."""
    import oracle
    oc = oracle.OracleCache(wl)
    q = oracle.to_numpy_bits(wl.queries())
    kpool, vpool = oc.k, oc.v
    if getattr(wl, "kv_format", "native") == "fp8":  # attention over the dequantised pages
        from oracle import fp8
        kpool, vpool = fp8.dequantized_pools(*fp8.fp8_pools_from(oc.k, oc.v))
        q = oracle.bits_to_f64(q)
    t_budget = seconds
    if wl.kind == "decode":
        # sequences in batch order until ~t_budget of work, measured by doing it
        done_bytes, elapsed, done = 0, 0.0, 0
        per_tok = wl.logical_bytes_per_token()
        while done < wl.num_seqs or elapsed < t_budget:
            s = done % wl.num_seqs
            rows = [(s, g) for g in range(wl.num_q_heads)]
            t0 = time.perf_counter()
            oracle.decode(kpool, vpool, q, oc.tables, wl.total_lens, wl.scale, rows=rows)
            elapsed += time.perf_counter() - t0
            n = int(wl.total_lens[s])
            done_bytes += (n * per_tok + wl.num_q_heads * wl.head_dim * (wl.elem_bytes + 4)
                           + 4 * (-(-n // wl.block_size)) + 4)
            done += 1
        return {"value": done_bytes / elapsed / 1e9, "unit": "GB/s", "cores": oracle.num_threads(),
                "kind": "oracle",
                "sample": "float64 oracle decode, %d sequence passes over the %d-sequence batch "
                          "(all %d q-heads each), %.1f s" % (done, wl.num_seqs, wl.num_q_heads,
                                                           elapsed),
                "seconds": elapsed, "tokens_per_s": done / elapsed}
    # prefill: a sample of (token, head) rows, scaled to TFLOP/s of visible work
    cu = np.concatenate([[0], np.cumsum(wl.new_lens)])
    rng = np.random.default_rng(0)
    T = int(cu[-1])
    rows, flops, elapsed = [], 0.0, 0.0
    while elapsed < t_budget and len(rows) < 1 << 16:
        batch = [(int(t), int(h)) for t, h in zip(rng.integers(0, T, 64),
                                                  rng.integers(0, wl.num_q_heads, 64))]
        t0 = time.perf_counter()
        oracle.prefill(oc.k, oc.v, q, cu, wl.total_lens, oc.tables, wl.scale, wl.causal, rows=batch)
        elapsed += time.perf_counter() - t0
        for t, h in batch:
            s = int(np.searchsorted(cu, t, side="right") - 1)
            pos = int(wl.cached_lens[s]) + (t - int(cu[s]))
            flops += 4.0 * wl.head_dim * (pos + 1)
        rows += batch
    return {"value": flops / elapsed / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": "float64 oracle prefill of %d random (token, q-head) rows, %.1f s"
                      % (len(rows), elapsed), "seconds": elapsed}


def reference_steps(wl, warmup: int, steps: int, budget_s: float):
    """The oracle as the reference arm: each step decodes one sequence of the
    batch (all q-heads) in float64, cycling through the batch; the timed steps
    stop early if the time budget runs out."""
    import oracle
    oc = oracle.OracleCache(wl)
    q = oracle.to_numpy_bits(wl.queries())
    kpool, vpool = oc.k, oc.v
    if getattr(wl, "kv_format", "native") == "fp8":  # attention over the dequantised pages
        from oracle import fp8
        kpool, vpool = fp8.dequantized_pools(*fp8.fp8_pools_from(oc.k, oc.v))
        q = oracle.bits_to_f64(q)
    per_tok = wl.logical_bytes_per_token()
    if wl.kind != "decode":
        r = cpu_oracle_run(wl, min(budget_s, 30.0))
        r.update({"steps": 1, "ms_per_step": r["seconds"] * 1e3})
        return r
    def one(s):
        rows = [(s, g) for g in range(wl.num_q_heads)]
        oracle.decode(kpool, vpool, q, oc.tables, wl.total_lens, wl.scale, rows=rows)
        n = int(wl.total_lens[s])
        return (n * per_tok + wl.num_q_heads * wl.head_dim * (wl.elem_bytes + 4)
                + 4 * (-(-n // wl.block_size)) + 4)
    for i in range(warmup):
        one(i % wl.num_seqs)
    done, nbytes, t0 = 0, 0, time.perf_counter()
    while done < max(1, steps) and time.perf_counter() - t0 < budget_s:
        nbytes += one((warmup + done) % wl.num_seqs)
        done += 1
    el = time.perf_counter() - t0
    return {"value": nbytes / el / 1e9, "unit": "GB/s", "cores": oracle.num_threads(),
            "steps": done, "ms_per_step": el / done * 1e3,
            "sample": "float64 oracle, one sequence (all %d q-heads) per step, %d steps in %.1f s"
                      % (wl.num_q_heads, done, el)}


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The slowest rank's time (one all-reduce, outside any timed region)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(bytes_per_rank: int, world: int, max_ms: float) -> float:
    """Whole-job GB/s: every rank's bytes over the slowest rank's step time."""
    return world * bytes_per_rank / (max_ms * 1e-3) / 1e9


# --------------------------------------------------------------------------- GPU arm
L2_BYTES = 129 * 10**6
HEADLINE = "decode_mha"
SUITE = ["decode_tiny", "decode_gqa", "decode_long_shared", "decode_long_shared_fp8", "prefill"]
DECODE_PATH = {"split": "split: pa_write_kv + pa_decode_partial + pa_decode_merge",
               "fused": "fused: pa_decode_step (new-token write, attention and split-KV merge in "
                        "one launch)",
               "window": "pa_write_kv + pa_decode_window (partition + merge)",
               "shared": "pa_write_kv + pa_decode_shared (shared-prefix pair units + own "
                         "partitions, then the merge)"}


def _events(torch, n, k):
    return [[torch.cuda.Event(enable_timing=True) for _ in range(k)] for _ in range(n)]


def _needs_flush(args, step_bytes: int) -> bool:
    """Flush L2 between timed steps when asked, or when one step's bytes would
    not push the previous step's data out of the 129 MB L2 by themselves."""
    return args.l2 == "flush" or step_bytes < 2 * L2_BYTES


def _l2_note(flush: bool, step_bytes: int) -> str:
    if flush:
        return ("flushed before every timed step by a 256 MiB write and a read of the same "
                "buffer, outside the step's events")
    return ("no flush: inputs larger than L2 (one step moves %.0f MB, L2 is 129 MB)"
            % (step_bytes / 1e6))


def _shared_inputs(torch, wl, dev):
    """partner / shared_lens of the workload's declared pairs (whole shared pages)."""
    B = wl.num_seqs
    partner = np.full(B, -1, np.int32)
    shared = np.zeros(B, np.int32)
    if wl.pair_of is not None:
        for s in range(B):
            q = int(wl.pair_of[s])
            if q >= 0:
                partner[s] = q
                shared[s] = int(wl.prefix_len[s]) // wl.block_size * wl.block_size
    return (torch.from_numpy(partner).to(dev), torch.from_numpy(shared).to(dev))


def bench_attention(args, wl, dev, world, mode="split", e2e=False, g=None):
    """One configuration: loop A times whole steps (value, ms_per_step, clocks),
    loop B puts an event between the kernels of each step (kernel_ms, the
    roofline of the dominant kernel).  Returns the record and the workload."""
    import torch
    import paged_kv_cache_148_gb300 as pkv
    from harness import GpuWorkload

    if g is None:
        g = GpuWorkload(wl, device=dev)
        if args.partition_tokens:
            g.set_partition_tokens(args.partition_tokens)
    stream = torch.cuda.current_stream(dev)
    is_decode = wl.kind == "decode"
    window = args.window if (is_decode and mode == "window") else 0
    if window > 0:
        g.set_window(window)
    fused = is_decode and mode == "fused"
    shared = None
    if is_decode and mode == "shared":
        partner, shared_lens = _shared_inputs(torch, wl, dev)
        ws_bytes = pkv.decode_shared_workspace_bytes(g.cache.pool, wl.num_seqs, wl.num_q_heads,
                                                     g.max_context, g.partition_tokens)
        shared = (partner, shared_lens, torch.empty(max(ws_bytes, 16), dtype=torch.uint8,
                                                    device=dev))
    max_parts = g.max_parts()
    if is_decode and mode == "shared":
        # the shared-prefix plan sizes its own partitions; its workspace holds
        # (max, sum, D values) floats per (sequence, q-head, partition slot)
        max_parts = ws_bytes // (wl.num_seqs * wl.num_q_heads * (wl.head_dim + 2) * 4)
    ab = algorithmic_bytes(wl, window)
    step_bytes = ab["decode_total"] + ab["write"] if is_decode else ab["kv"] + ab["q"] + ab["out"]
    do_flush = _needs_flush(args, step_bytes)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev) if do_flush else None

    def attend():
        if shared is not None:
            pkv.decode_shared(g.cache.pool, g.q, g.block_tables, g.context_lens, g.max_context,
                              shared[0], shared[1], wl.scale, out=g.out, workspace=shared[2],
                              partition_tokens=g.partition_tokens, d_err=g.err, stream=stream)
        else:
            g.attend(stream)

    # kernels of one step, in launch order (events go between them in loop B)
    if fused:
        phases = [("decode_step", lambda: g.step(stream, fused=True))]
    elif is_decode and mode == "split":
        phases = [("write_kv", lambda: g.write_new(stream)),
                  ("decode_partition", lambda: g.attend(stream, "partial")),
                  ("decode_merge", lambda: g.attend(stream, "merge"))]
    elif is_decode:
        phases = [("write_kv", lambda: g.write_new(stream)),
                  ("decode_%s (partition + merge)" % mode, attend)]
    else:
        phases = [("write_kv", lambda: g.write_new(stream)), ("prefill", attend)]

    def step():
        for _, fn in phases:
            fn()

    for i in range(args.warmup):
        if do_flush:
            flush_l2(flush, i)
        step()
    torch.cuda.synchronize(dev)
    g.err.zero_()
    K = args.steps
    ev = _events(torch, K, 2)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    for i in range(K):
        if do_flush:
            flush_l2(flush, i)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    step_ms = np.array([a.elapsed_time(b) for a, b in ev])
    KB = min(K, 500)
    evk = _events(torch, KB, len(phases) + 1)
    torch.cuda.synchronize(dev)
    for i in range(KB):
        if do_flush:
            flush_l2(flush, i)
        e = evk[i]
        e[0].record(stream)
        for j, (_, fn) in enumerate(phases):
            fn()
            e[j + 1].record(stream)
    torch.cuda.synchronize(dev)
    err = int(g.err.item())
    if err:
        raise RuntimeError("%s: device error during the timed loops: %s"
                           % (wl.name, pkv.status_str(err)))
    kernel_ms = {name: float(np.mean([e[j].elapsed_time(e[j + 1]) for e in evk]))
                 for j, (name, _) in enumerate(phases)}
    ms = max_over_ranks(float(step_ms.mean()), world, dev)
    hbm_peak, tf_peak, peak_src = measured_peaks()
    rec = {"workload": wl.name, "steps": K, "ms_per_step": ms, "kernel_ms": kernel_ms,
           "clocks": clk, "l2": _l2_note(do_flush, step_bytes),
           "dtype": ("e4m3 pages (float32 row scales), bf16 queries, f32 arithmetic"
                     if getattr(wl, "kv_format", "native") == "fp8" else wl.dtype)}
    cfg = {"workload": wl.name, "num_seqs": wl.num_seqs, "num_q_heads": wl.num_q_heads,
           "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
           "block_size": wl.block_size, "num_blocks": wl.num_blocks,
           "context_lens": "sum %d, min %d, max %d" % (int(wl.total_lens.sum()),
                                                      int(wl.total_lens.min()),
                                                      int(wl.total_lens.max())),
           "per_rank": "each rank runs its own copy of the batch (independent replicas)",
           "l2": rec["l2"]}
    if is_decode:
        cfg.update({"split_kv_partitions_max": max_parts, "window": window or "none",
                    "path": DECODE_PATH[mode], "partition_tokens": args.partition_tokens or "auto",
                    "kernel": kernel_name(wl, mode)})
        phys = physical_kv_bytes(wl, g.tables_list(), window)
        cfg["kv_bytes"] = {"logical": ab["kv"], "unique_physical": phys,
                           "counted": "logical (each sequence's pages once per sequence)"}
        per_rank = ab["decode_total"]
        rec.update({"value": aggregate_value(per_rank, world, ms), "unit": "GB/s",
                    "tokens_per_s": world * wl.num_seqs / (ms * 1e-3),
                    "pct_of_hbm_peak": 100.0 * (per_rank / (ms * 1e-3) / 1e9) / hbm_peak,
                    "pct_of_nominal_8tbs": 100.0 * (per_rank / (ms * 1e-3) / 1e9) / 8000.0})
        if ab["kv"] != phys:
            rec["value_physical"] = aggregate_value(per_rank - ab["kv"] + phys, world, ms)
        dom = "decode_step" if fused else ("decode_partition" if mode == "split" else phases[-1][0])
        launch_ms = kernel_ms[dom]
        achieved = per_rank / (launch_ms * 1e-3) / 1e9
        kname = kernel_name(wl, mode)
        rec["roofline"] = {"kernel": kname, "bound": "hbm", "achieved": achieved,
                           "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                           "peak_source": peak_src + " hbm_gbs (copy, burst)",
                           "traffic": recorded_traffic(kname, wl.name + ("" if mode == "split"
                                                                         else "_" + mode)),
                           "algorithmic_bytes": per_rank, "launch_ms": launch_ms,
                           "timed": "%s%s" % (dom, "" if mode == "split" else
                                              " (all of its kernels)")}
        # write + partition kernel, + the merge when a context spans partitions
        # (the shared-prefix plan always has room for one more slot, so it merges)
        if fused:
            launches = K
        else:
            launches = K * (2 + (1 if (max_parts > 1 or mode == "shared") else 0))
    else:
        flops = prefill_flops(wl)
        rec.update({"value": world * flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "tokens_per_s": world * int(wl.new_lens.sum()) / (ms * 1e-3)})
        pf_ms = kernel_ms["prefill"]
        achieved = flops / (pf_ms * 1e-3) / 1e12
        rec["roofline"] = {"kernel": "prefill_kernel", "bound": "tensor", "achieved": achieved,
                           "peak": tf_peak, "unit": "TFLOP/s", "frac": achieved / tf_peak,
                           "peak_source": peak_src + " bf16_tflops (burst)",
                           "traffic": recorded_traffic("prefill_kernel", wl.name),
                           "algorithmic_flops": flops, "launch_ms": pf_ms}
        cfg["path"] = "pa_write_kv + pa_prefill"
        launches = K * 2
    rec["gpu_launches"] = launches
    rec["config"] = cfg
    if e2e:
        rec["e2e"] = run_e2e(args, g, stream, dev, is_decode, fused)
    return rec, g


def kernel_name(wl, mode="split") -> str:
    """The library kernel that dominates a decode step of this workload."""
    if wl.kind != "decode":
        return "prefill_kernel"
    if mode == "fused":
        return "decode_step"
    if mode == "shared":
        return "decode_shared_kernel"
    G = wl.num_q_heads // wl.num_kv_heads
    fmt = getattr(wl, "kv_format", "native")
    if (wl.dtype == "bf16" and fmt == "native" and wl.head_dim == 128 and wl.block_size >= 16
            and G in (2, 4, 8)):
        return "decode_mma_kernel"
    if fmt == "fp8" and wl.head_dim == 128 and wl.block_size >= 16 and G == 8:
        return "decode_fp8_mma_kernel"
    return "decode_partition_kernel"


def bench_write(args, wl, dev, world):
    """pa_write_kv of one prefill batch's new rows (8192 rows of K and V)."""
    import torch
    from harness import GpuWorkload
    g = GpuWorkload(wl, device=dev)
    stream = torch.cuda.current_stream(dev)
    ab = algorithmic_bytes(wl)
    return _micro(args, dev, world, "write_kv_kernel", ab["write"],
                  lambda: g.write_new(stream), g.err,
                  {"workload": wl.name + " new rows", "rows": int(wl.new_lens.sum()),
                   "row_bytes": wl.num_kv_heads * wl.head_dim * wl.elem_bytes,
                   "bytes": "K and V rows read and written + 8-byte slots"})


def bench_copy(args, dev, world):
    """pa_copy_blocks of 10% of a decode_gqa-shaped pool, random src != dst."""
    import torch
    import paged_kv_cache_148_gb300 as pkv
    wl = workloads.decode_gqa()
    pool = pkv.KVPool(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim,
                      wl.torch_dtype, dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(3)
    for t in (pool.k, pool.v):
        t.view(torch.int16).random_(generator=gen)
    rng = np.random.default_rng(1102)
    n = wl.num_blocks // 10
    ids = rng.permutation(wl.num_blocks)
    src = torch.from_numpy(ids[:n].astype(np.int32)).to(dev)
    dst = torch.from_numpy(ids[n:2 * n].astype(np.int32)).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    page = wl.num_kv_heads * wl.block_size * wl.head_dim * wl.elem_bytes
    nbytes = 2 * n * page * 2 + 2 * n * 4
    rec = _micro(args, dev, world, "copy_blocks_kernel", nbytes,
                 lambda: pkv.copy_blocks(pool, src, dst, d_err=err, stream=stream), err,
                 {"workload": "decode_gqa-shaped pool (%d blocks), %d pairs" % (wl.num_blocks, n),
                  "page_bytes": page,
                  "bytes": "K and V pages read and written + 8 bytes of ids per pair"})
    del pool
    return rec


def _micro(args, dev, world, kname, nbytes, fn, err, cfg):
    import torch
    import paged_kv_cache_148_gb300 as pkv
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for i in range(max(args.warmup, 3)):
        flush_l2(flush, i)
        fn()
    torch.cuda.synchronize(dev)
    err.zero_()
    K = args.steps
    ev = _events(torch, K, 2)
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    for i in range(K):
        flush_l2(flush, i)
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    e = int(err.item())
    if e:
        raise RuntimeError("%s: device error: %s" % (kname, pkv.status_str(e)))
    ms = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in ev])), world, dev)
    hbm_peak, _, peak_src = measured_peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    cfg["l2"] = _l2_note(True, nbytes)
    return {"workload": cfg["workload"], "steps": K, "ms_per_step": ms, "value": world * gbs,
            "unit": "GB/s", "kernel_ms": {kname: ms}, "clocks": clk, "gpu_launches": K,
            "roofline": {"kernel": kname, "bound": "hbm", "achieved": gbs, "peak": hbm_peak,
                         "unit": "GB/s", "frac": gbs / hbm_peak,
                         "peak_source": peak_src + " hbm_gbs (copy, burst)",
                         "traffic": None, "algorithmic_bytes": nbytes, "launch_ms": ms},
            "config": cfg}


def run_ours(args, rank, world, local_rank):
    """The headline configuration (its record is the line's top level) and,
    for the default suite, one record per other configuration plus the
    shared-prefix decode and the write / copy microbenchmarks."""
    import torch
    import paged_kv_cache_148_gb300 as pkv

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    pkv.build()
    name = HEADLINE if args.workload == "suite" else args.workload
    mode = args.path if args.path != "split" else ("window" if args.window > 0 else "split")
    wl = (workloads.WORKLOADS[name]() if args.workload == "suite"
          else workloads.WORKLOADS[name](args.scale))
    head, g = bench_attention(args, wl, dev, world, mode, e2e=True)
    del g
    torch.cuda.empty_cache()
    res = {"metric": METRIC if wl.kind == "decode" else
           "paged chunked-prefill TFLOP/s (causal-visible) on 1 GB300",
           "value": head["value"], "unit": head["unit"], "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "data": "synthetic", "dtype": head["dtype"]}
    for k in ("tokens_per_s", "pct_of_hbm_peak", "pct_of_nominal_8tbs", "roofline",
              "kernel_ms", "gpu_launches", "e2e", "clocks", "config"):
        if k in head:
            res[k] = head[k]
    res["kernel_timing"] = ("kernel_ms and roofline.launch_ms come from a second loop of %d "
                            "steps with an event between every kernel" % min(args.steps, 500))
    if args.workload == "suite":
        suite = {}
        for other in SUITE:
            owl = workloads.WORKLOADS[other]()
            rec, g = bench_attention(args, owl, dev, world, "split")
            suite[other] = rec
            if other == "decode_long_shared":
                rec2, _ = bench_attention(args, owl, dev, world, "shared", g=g)
                suite["decode_long_shared (shared-prefix decode)"] = rec2
            if other == "prefill":
                suite["write_kv (prefill rows)"] = bench_write(args, owl, dev, world)
            del g
            torch.cuda.empty_cache()
        suite["copy_blocks (10% of a decode_gqa pool)"] = bench_copy(args, dev, world)
        torch.cuda.empty_cache()
        res["suite"] = suite
    return res, wl


def run_e2e(args, g, stream, dev, is_decode, fused=False):
    """The same step through the public API with pinned host buffers: every
    step copies its inputs host -> device and its output device -> host
    inside the timed region.  As a serving loop would, the uploads and the
    downloads run on their own streams against two sets of device buffers,
    so step i+1's inputs go up and step i's output comes down while the
    kernels of a step run; a set is reused only after the step that used it
    has been copied out."""
    import torch
    wl = g.wl
    names = ["q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens"]
    if not is_decode:
        names.append("cu_seqlens_q")
    host_in = {"q": g.q_host, "k_new": g.k_new_host, "v_new": g.v_new_host,
               "slot_mapping": torch.from_numpy(g.slot_mapping_host),
               "block_tables": g.block_tables.cpu(), "context_lens": g.context_lens.cpu()}
    if not is_decode:
        host_in["cu_seqlens_q"] = g.cu_seqlens_q.cpu()
    pinned = {k: host_in[k].contiguous().pin_memory() for k in names}
    own = {k: getattr(g, k) for k in names + ["out"]}
    sets = [own, {k: torch.empty_like(v) for k, v in own.items()}]
    out_host = [torch.empty(g.out.shape, dtype=g.out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = out_host[0].numel() * out_host[0].element_size()
    up_stream, down_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(n):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        up = [torch.cuda.Event() for _ in range(n)]
        done = [torch.cuda.Event() for _ in range(n)]
        down = [torch.cuda.Event() for _ in range(n)]
        start.record(stream)
        up_stream.wait_event(start)
        for i in range(n):
            k = i % 2
            with torch.cuda.stream(up_stream):
                if i >= 2:
                    up_stream.wait_event(down[i - 2])  # set k is free again
                for name in names:
                    sets[k][name].copy_(pinned[name], non_blocking=True)
                up[i].record(up_stream)
            stream.wait_event(up[i])
            for name, t in sets[k].items():
                setattr(g, name, t)
            g.step(stream, fused=fused)
            done[i].record(stream)
            with torch.cuda.stream(down_stream):
                down_stream.wait_event(done[i])
                out_host[k].copy_(sets[k]["out"], non_blocking=True)
                down[i].record(down_stream)
        stream.wait_event(down[n - 1])
        end.record(stream)
        return start, end

    try:
        run(3)
        torch.cuda.synchronize(dev)
        n = max(1, args.e2e_steps)
        start, end = run(n)
        torch.cuda.synchronize(dev)
    finally:
        for name, t in own.items():
            setattr(g, name, t)
    t = start.elapsed_time(end) / n
    if is_decode:
        val, unit = algorithmic_bytes(wl, g.window)["decode_total"] / (t * 1e-3) / 1e9, "GB/s"
    else:
        val, unit = prefill_flops(wl) / (t * 1e-3) / 1e12, "TFLOP/s"
    return {"value": val, "unit": unit, "ms_per_step": t, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": n,
            "copies": "pinned host buffers; inputs up and output down every step on their "
                      "own streams, double-buffered against the compute stream"}


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus if args.gpus == 1 else 1)))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        wl = workloads.WORKLOADS[HEADLINE if args.workload == "suite" else args.workload]()
        cpu = reference_steps(wl, args.warmup, args.steps, budget_s=150.0)
        line = {"impl": "reference", "metric": METRIC if wl.kind == "decode" else
                "paged chunked-prefill TFLOP/s (causal-visible) on 1 GB300",
                "value": cpu["value"], "unit": cpu["unit"], "higher_is_better": True,
                "n_gpus": world, "steps": cpu["steps"], "warmup": args.warmup,
                "ms_per_step": cpu["ms_per_step"], "data": "synthetic", "dtype": "f64",
                "scaling": "weak", "vs_baseline": None, "config": {"workload": wl.name},
                "cpu_baseline": {"value": cpu["value"], "unit": cpu["unit"], "cores": cpu["cores"],
                                 "kind": "oracle", "sample": cpu["sample"]},
                "e2e": {"value": cpu["value"], "unit": cpu["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl")
    res, wl = run_ours(args, rank, world, local_rank)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_run(wl, args.cpu_seconds)
        res["cpu_baseline"] = {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")}
    elif rank == 0:
        res["cpu_baseline"] = None
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(res))
    return 0


if __name__ == "__main__":
    sys.exit(main())

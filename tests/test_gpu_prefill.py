"""GPU parity of pa_prefill (tcgen05 tensor-core path) against the float64 oracle.

Tolerance for bf16 operands with fp32 accumulation and fp32 output:
max |err| <= 2e-3 and relative L2 <= 1e-3 (P is rounded to bf16 before the
P*V product, as on the tensor cores; the oracle keeps it in float64).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_148_gb300 as pkv
import workloads
from harness import GpuWorkload

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pkv.build()
    yield
    torch.cuda.synchronize()


def _check(got, ref, what):
    got = np.asarray(got, np.float64)
    assert np.isfinite(got).all(), what + ": non-finite output"
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err <= MAX_ABS and rel <= REL_L2, "%s: max abs %.3g rel L2 %.3g" % (what, err, rel)


def _run(wl, rows=None):
    g = GpuWorkload(wl)
    g.err.zero_()
    out = g.step()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0, pkv.status_str(int(g.err.item()))
    oc = oracle.OracleCache(wl)
    cu = np.concatenate([[0], np.cumsum(wl.new_lens)])
    q = oracle.to_numpy_bits(g.q_host)
    ref = oracle.prefill(oc.k, oc.v, q, cu, wl.total_lens, oc.tables, wl.scale,
                         causal=wl.causal, rows=rows)
    got = out.cpu().numpy()
    if rows is not None:
        got = np.stack([got[t, h] for t, h in rows])
    return got, ref


def test_prefill_single_tile():
    wl = workloads.custom_decode(1, 4, 1, 128, 16, "bf16", [0], seed=1, new_lens=[32],
                                 kind="prefill")
    got, ref = _run(wl)
    _check(got, ref, "single tile")


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_prefill_group_sizes(G):
    wl = workloads.custom_decode(3, 2 * G, 2, 128, 16, "bf16", [100, 0, 257], seed=G,
                                 new_lens=[70, 129, 40], kind="prefill")
    got, ref = _run(wl)
    _check(got, ref, "G=%d" % G)


@pytest.mark.parametrize("block_size", [8, 16, 32, 64, 128])
def test_prefill_block_sizes(block_size):
    wl = workloads.custom_decode(2, 8, 2, 128, block_size, "bf16", [300, 77], seed=block_size,
                                 new_lens=[50, 200], kind="prefill")
    got, ref = _run(wl)
    _check(got, ref, "bp=%d" % block_size)


def test_prefill_non_causal():
    wl = workloads.custom_decode(2, 8, 2, 128, 16, "bf16", [130, 5], seed=11, new_lens=[33, 64],
                                 kind="prefill", causal=False)
    got, ref = _run(wl)
    _check(got, ref, "non-causal")


def test_prefill_ragged_lengths():
    cached = [0, 1, 15, 16, 17, 127, 128, 129, 500]
    new = [1, 2, 31, 32, 33, 97, 128, 5, 300]
    wl = workloads.custom_decode(len(cached), 8, 2, 128, 16, "bf16", cached, seed=13,
                                 new_lens=new, kind="prefill")
    got, ref = _run(wl)
    _check(got, ref, "ragged")


def test_prefill_scaled_workload():
    wl = workloads.prefill(scale=1 / 8)
    got, ref = _run(wl)
    _check(got, ref, wl.name)


def test_prefill_full_size_sampled_rows():
    wl = workloads.prefill()
    rng = np.random.default_rng(5)
    T = int(wl.new_lens.sum())
    rows = [(int(t), int(h)) for t, h in zip(rng.integers(0, T, 160),
                                             rng.integers(0, wl.num_q_heads, 160))]
    rows += [(0, 0), (T - 1, wl.num_q_heads - 1), (511, 3), (512, 31)]
    got, ref = _run(wl, rows=rows)
    _check(got, ref, "prefill full size")


def test_prefill_flags_table_entry_outside_pool():
    wl = workloads.custom_decode(2, 8, 2, 128, 16, "bf16", [40, 40], seed=17, new_lens=[8, 8],
                                 kind="prefill")
    g = GpuWorkload(wl)
    g.write_new()
    bt = g.block_tables.clone()
    bt[1, 0] = wl.num_blocks + 1
    g.err.zero_()
    pkv.prefill(g.cache.pool, g.q, g.cu_seqlens_q, g.context_lens, bt, g.max_q, g.max_context,
                wl.scale, out=g.out, d_err=g.err)
    torch.cuda.synchronize()
    assert int(g.err.item()) == pkv.PA_ERR_OUT_OF_RANGE

"""GPU parity of pa_decode_step (the new token of every sequence written and
attended in one launch, split-KV partials merged by the last partition of each
(sequence, kv-head)) against the float64 oracle.

  - the pool after the step: bit-exact against the oracle's writes;
  - bf16 output: max |err| <= 2e-3 and relative L2 <= 1e-3; fp32: <= 1e-5;
  - the per-(sequence, kv-head) semaphores are zero again after every call.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_148_gb300 as pkv
import workloads
from harness import GpuWorkload

pytestmark = pytest.mark.gpu

BF16_MAX_ABS, BF16_REL_L2, F32_MAX_ABS = 2e-3, 1e-3, 1e-5


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pkv.build()
    pkv.lib()
    yield
    torch.cuda.synchronize()


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.uint8).numpy().reshape(-1)


def _close(got, ref, dtype, what):
    got = np.asarray(got, np.float64)
    assert np.isfinite(got).all(), "%s: non-finite output" % what
    err = np.abs(got - ref).max()
    if dtype == "f32":
        assert err <= F32_MAX_ABS, "%s max abs err %.3g" % (what, err)
    else:
        rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
        assert err <= BF16_MAX_ABS and rel <= BF16_REL_L2, "%s: max abs %.3g rel L2 %.3g" % (
            what, err, rel)


def _semaphores_zero(g):
    ws = g.step_workspace
    if ws is None:
        return True
    n = g.wl.num_seqs * g.wl.num_kv_heads * 4
    return bool((ws[-n:] == 0).all().item())


def _step_and_check(wl, part=0, rows=None):
    g = GpuWorkload(wl)
    if part:
        g.set_partition_tokens(part)
    g.err.zero_()
    out = g.step(fused=True)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0, pkv.status_str(int(g.err.item()))
    assert _semaphores_zero(g)
    oc = oracle.OracleCache(wl)
    assert np.array_equal(_bits(g.cache.pool.k), oc.k.view(np.uint8).reshape(-1))
    assert np.array_equal(_bits(g.cache.pool.v), oc.v.view(np.uint8).reshape(-1))
    q = oracle.to_numpy_bits(g.q_host)
    got = out.cpu().numpy()
    if rows is None:
        ref = oracle.decode(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale)
    else:
        ref = oracle.decode(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale, rows=rows)
        got = np.stack([got[s, h] for s, h in rows])
    return g, got, ref


CASES = [
    ("tiny", lambda: workloads.decode_tiny()),
    ("gqa_small", lambda: workloads.decode_gqa(scale=1 / 8)),
    ("mha_small", lambda: workloads.decode_mha(scale=1 / 8)),
    ("long_shared_small", lambda: workloads.decode_long_shared(scale=1 / 64)),
]


@pytest.mark.parametrize("name,make", CASES)
def test_decode_step_matches_oracle(name, make):
    wl = make()
    g, got, ref = _step_and_check(wl)
    _close(got, ref, wl.dtype, name)


@pytest.mark.parametrize("part", [16, 32, 48, 256, 1 << 20])
def test_decode_step_partition_sizes(part):
    # many partitions merged in-kernel, uneven ones, and a single partition
    wl = workloads.decode_gqa(scale=1 / 16)
    g, got, ref = _step_and_check(wl, part=part)
    _close(got, ref, wl.dtype, "part=%d" % part)


EDGE_LENS = [0, 1, 14, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 129, 300]


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("block_size", [1, 4, 16, 64])
def test_decode_step_edge_lengths_bf16(G, block_size):
    wl = workloads.custom_decode(len(EDGE_LENS), 2 * G, 2, 128, block_size, "bf16", EDGE_LENS,
                                 seed=G * 1000 + block_size)
    for part in (0, 32):
        g, got, ref = _step_and_check(wl, part=part)
        _close(got, ref, "bf16", "G=%d bp=%d part=%d" % (G, block_size, part))


@pytest.mark.parametrize("G", [1, 4])
def test_decode_step_edge_lengths_f32(G):
    wl = workloads.custom_decode(len(EDGE_LENS), 2 * G, 2, 64, 4, "f32", EDGE_LENS, seed=G + 7)
    g, got, ref = _step_and_check(wl, part=48)
    _close(got, ref, "f32", "G=%d" % G)


def test_decode_step_repeated_calls_and_cuda_graph():
    wl = workloads.decode_gqa(scale=1 / 16)
    g = GpuWorkload(wl)
    g.set_partition_tokens(32)  # several partitions per sequence: the in-kernel merge runs
    outs = []
    for _ in range(3):  # re-writing the same token gives the same result every time
        g.err.zero_()
        outs.append(g.step(fused=True).clone())
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    assert _semaphores_zero(g)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    # the same step captured into a CUDA graph and replayed
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g.step(fused=True, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    g.out.zero_()
    with torch.cuda.graph(graph):
        g.step(fused=True, stream=torch.cuda.current_stream())
    for _ in range(2):
        g.out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(g.out, outs[0])
    assert _semaphores_zero(g)
    assert int(g.err.item()) == 0


def test_decode_step_flags_a_slot_that_is_not_the_last_position():
    wl = workloads.decode_gqa(scale=1 / 16)
    g = GpuWorkload(wl)
    before_k = _bits(g.cache.pool.k).copy()
    bad = g.slot_mapping.clone()
    bad[0] = g.slot_mapping[1]          # a valid slot of another sequence
    bad[2] = wl.num_blocks * wl.block_size  # outside the pool
    g.err.zero_()
    pkv.decode_step(g.cache.pool, g.k_new, g.v_new, bad, g.q, g.block_tables, g.context_lens,
                    g.max_context, wl.scale, g.step_workspace, out=g.out, d_err=g.err)
    torch.cuda.synchronize()
    assert int(g.err.item()) in (pkv.PA_ERR_INVALID_ARG, pkv.PA_ERR_OUT_OF_RANGE)
    assert _semaphores_zero(g)
    # rows 0 and 2 not written, the others written as the oracle writes them
    oc = oracle.OracleCache(wl, write_new=False)
    keep = [s for s in range(wl.num_seqs) if s not in (0, 2)]
    oracle.write_kv(oc.k, oc.v, oracle.to_numpy_bits(g.k_new_host[keep]),
                    oracle.to_numpy_bits(g.v_new_host[keep]), g.slot_mapping_host[keep])
    assert np.array_equal(_bits(g.cache.pool.k), oc.k.view(np.uint8).reshape(-1))
    assert not np.array_equal(before_k, _bits(g.cache.pool.k))


@pytest.mark.parametrize("make", [workloads.decode_gqa, workloads.decode_long_shared],
                         ids=["decode_gqa", "decode_long_shared"])
def test_decode_step_full_size(make):
    wl = make()
    rng = np.random.default_rng(21)
    rows = [(int(s), int(h)) for s, h in zip(rng.integers(0, wl.num_seqs, 64),
                                             rng.integers(0, wl.num_q_heads, 64))]
    g, got, ref = _step_and_check(wl, rows=rows)
    _close(got, ref, wl.dtype, wl.name + " sampled")

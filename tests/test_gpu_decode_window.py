"""GPU parity of pa_decode_window (sliding-window paged decode: the query at
position n-1 attends to positions max(0, n-w)..n-1) against the float64
oracle's orc_decode_window.  Tolerances as for pa_decode: bf16 max |err| <=
2e-3 and relative L2 <= 1e-3, fp32 max |err| <= 1e-5."""
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


def _run(wl, window, part=0, rows=None):
    g = GpuWorkload(wl)
    g.set_window(window)
    if part:
        g.set_partition_tokens(part)
    g.err.zero_()
    out = g.step()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0, pkv.status_str(int(g.err.item()))
    oc = oracle.OracleCache(wl)
    q = oracle.to_numpy_bits(g.q_host)
    got = out.cpu().numpy()
    if rows is None:
        ref = oracle.decode_window(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale, window)
    else:
        ref = oracle.decode_window(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale, window,
                                   rows=rows)
        got = np.stack([got[s, h] for s, h in rows])
    return g, got, ref


@pytest.mark.parametrize("window", [1, 15, 16, 17, 100, 1000, 1 << 20])
def test_window_decode_matches_oracle(window):
    wl = workloads.decode_gqa(scale=1 / 8)
    g, got, ref = _run(wl, window)
    _close(got, ref, wl.dtype, "w=%d" % window)


@pytest.mark.parametrize("part", [16, 32, 48, 256])
def test_window_partition_sizes(part):
    wl = workloads.decode_gqa(scale=1 / 16)
    g, got, ref = _run(wl, 300, part=part)
    _close(got, ref, wl.dtype, "part=%d" % part)


EDGE_LENS = [0, 1, 14, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 129, 300]


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("block_size", [1, 4, 16, 64])
def test_window_edge_lengths_bf16(G, block_size):
    wl = workloads.custom_decode(len(EDGE_LENS), 2 * G, 2, 128, block_size, "bf16", EDGE_LENS,
                                 seed=G * 31 + block_size)
    for window, part in ((1, 0), (17, 0), (33, 16), (64, 32)):
        g, got, ref = _run(wl, window, part=part)
        _close(got, ref, "bf16", "G=%d bp=%d w=%d part=%d" % (G, block_size, window, part))


def test_window_f32_tiny():
    wl = workloads.decode_tiny()
    for window in (1, 5, 16, 40):
        g, got, ref = _run(wl, window)
        _close(got, ref, "f32", "w=%d" % window)


def test_pages_before_the_window_are_not_read():
    # table entries wholly before the window point outside the pool: a read of
    # any of them would be flagged; the windowed result stays exact
    wl = workloads.decode_gqa(scale=1 / 16)
    g = GpuWorkload(wl)
    window = 100
    g.set_window(window)
    g.write_new()
    bt = g.block_tables.clone()
    lens = g.context_lens.cpu().numpy()
    for s, n in enumerate(lens):
        first_page = max(0, int(n) - window) // wl.block_size
        bt[s, :first_page] = wl.num_blocks + 7
    g.err.zero_()
    out = pkv.decode_window(g.cache.pool, g.q, bt, g.context_lens, g.max_context, window,
                            wl.scale, workspace=g.workspace, d_err=g.err)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    oc = oracle.OracleCache(wl)
    ref = oracle.decode_window(oc.k, oc.v, oracle.to_numpy_bits(g.q_host), oc.tables,
                               wl.total_lens, wl.scale, window)
    _close(out.cpu().numpy(), ref, wl.dtype, "poisoned prefix")


def test_window_must_be_positive():
    wl = workloads.decode_tiny()
    g = GpuWorkload(wl)
    with pytest.raises(pkv.PagedKVError):
        pkv.decode_window(g.cache.pool, g.q, g.block_tables, g.context_lens, g.max_context, 0,
                          wl.scale)


def test_window_full_size_long_context():
    wl = workloads.decode_long_shared()
    rng = np.random.default_rng(33)
    rows = [(int(s), int(h)) for s, h in zip(rng.integers(0, wl.num_seqs, 48),
                                             rng.integers(0, wl.num_q_heads, 48))]
    g, got, ref = _run(wl, 4096, rows=rows)
    _close(got, ref, wl.dtype, "long context w=4096")

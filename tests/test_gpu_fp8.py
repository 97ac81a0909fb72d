"""GPU parity of FP8 (E4M3) pages: pa_write_kv quantises bf16 rows into codes
and row scales bit-exactly as the oracle (oracle/fp8.py) does, pa_copy_blocks
carries the scales, and pa_decode / pa_decode_window over the pages match the
float64 oracle over the dequantised values (bf16 tolerances: max |err| <= 2e-3,
relative L2 <= 1e-3)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_148_gb300 as pkv
import workloads
from harness import GpuWorkload
from oracle import fp8

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pkv.build()
    pkv.lib()
    yield
    torch.cuda.synchronize()


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.uint8).numpy().reshape(-1)


def _close(got, ref, what):
    got = np.asarray(got, np.float64)
    assert np.isfinite(got).all(), "%s: non-finite output" % what
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err <= MAX_ABS and rel <= REL_L2, "%s: max abs %.3g rel L2 %.3g" % (what, err, rel)


def _oracle_fp8(wl):
    oc = oracle.OracleCache(wl)
    kc, vc, ks, vs = fp8.fp8_pools_from(oc.k, oc.v)
    return oc, kc, vc, ks, vs


def _reference(wl, g, oc, kc, vc, ks, vs, window=0, rows=None):
    kd, vd = fp8.dequantized_pools(kc, vc, ks, vs)
    q = oracle.bits_to_f64(oracle.to_numpy_bits(g.q_host))
    if window:
        return oracle.decode_window(kd, vd, q, oc.tables, wl.total_lens, wl.scale, window,
                                    rows=rows)
    return oracle.decode(kd, vd, q, oc.tables, wl.total_lens, wl.scale, rows=rows)


WRITE_CASES = [
    ("gqa", lambda: workloads.decode_gqa(scale=1 / 8)),
    ("long_shared", lambda: workloads.decode_long_shared(scale=1 / 256)),
    ("bp4", lambda: workloads.custom_decode(6, 8, 2, 128, 4, "bf16", [0, 3, 4, 17, 40, 99])),
]


@pytest.mark.parametrize("name,make", WRITE_CASES)
def test_fp8_pages_written_and_copied_bit_exact(name, make):
    wl = workloads.with_fp8_pages(make())
    g = GpuWorkload(wl)
    g.err.zero_()
    g.write_new()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    oc, kc, vc, ks, vs = _oracle_fp8(wl)
    assert g.tables_list() == oc.tables and g.cow_pairs == oc.cow_pairs
    pool = g.cache.pool
    assert np.array_equal(_bits(pool.k), kc.reshape(-1))
    assert np.array_equal(_bits(pool.v), vc.reshape(-1))
    assert np.array_equal(_bits(pool.k_scale), ks.view(np.uint8).reshape(-1))
    assert np.array_equal(_bits(pool.v_scale), vs.view(np.uint8).reshape(-1))


DECODE_CASES = [
    ("gqa", lambda: workloads.decode_gqa(scale=1 / 8), 0),
    ("gqa_parts", lambda: workloads.decode_gqa(scale=1 / 16), 32),
    ("mha", lambda: workloads.decode_mha(scale=1 / 16), 0),
    ("long_shared", lambda: workloads.decode_long_shared(scale=1 / 64), 0),
]


@pytest.mark.parametrize("name,make,part", DECODE_CASES)
def test_fp8_decode_matches_oracle(name, make, part):
    wl = workloads.with_fp8_pages(make())
    g = GpuWorkload(wl)
    if part:
        g.set_partition_tokens(part)
    g.err.zero_()
    out = g.step()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0, pkv.status_str(int(g.err.item()))
    _close(out.cpu().numpy(), _reference(wl, g, *_oracle_fp8(wl)), name)


EDGE_LENS = [0, 1, 14, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 129, 300]


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("block_size", [4, 8, 16, 64])
def test_fp8_decode_edge_lengths(G, block_size):
    wl = workloads.with_fp8_pages(workloads.custom_decode(
        len(EDGE_LENS), 2 * G, 2, 128, block_size, "bf16", EDGE_LENS, seed=G * 7 + block_size))
    for part, window in ((0, 0), (32, 0), (0, 33)):
        g = GpuWorkload(wl)
        if part:
            g.set_partition_tokens(part)
        if window:
            g.set_window(window)
        g.err.zero_()
        out = g.step()
        torch.cuda.synchronize()
        assert int(g.err.item()) == 0
        ref = _reference(wl, g, *_oracle_fp8(wl), window=window)
        _close(out.cpu().numpy(), ref, "G=%d bp=%d part=%d w=%d" % (G, block_size, part, window))


def test_fp8_limits_are_reported():
    wl = workloads.with_fp8_pages(workloads.custom_decode(3, 8, 2, 128, 2, "bf16", [5, 9, 20]))
    g = GpuWorkload(wl)
    g.write_new()
    with pytest.raises(pkv.PagedKVError) as e:  # 2-token blocks: scale pieces under 16 bytes
        g.attend()
    assert e.value.status == pkv.PA_ERR_UNSUPPORTED
    wl = workloads.with_fp8_pages(workloads.decode_gqa(scale=1 / 32))
    g = GpuWorkload(wl)
    with pytest.raises(pkv.PagedKVError) as e:  # the one-launch step writes raw rows
        g.step(fused=True)
    assert e.value.status == pkv.PA_ERR_UNSUPPORTED
    assert pkv.page_size_bytes(g.cache.pool) == 2 * 16 * 8 * (128 + 4)


def test_fp8_decode_full_size_sampled():
    wl = workloads.decode_gqa_fp8()
    g = GpuWorkload(wl)
    g.err.zero_()
    out = g.step()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    rng = np.random.default_rng(17)
    rows = [(int(s), int(h)) for s, h in zip(rng.integers(0, wl.num_seqs, 96),
                                             rng.integers(0, wl.num_q_heads, 96))]
    ref = _reference(wl, g, *_oracle_fp8(wl), rows=rows)
    got = out.cpu().numpy()
    _close(np.stack([got[s, h] for s, h in rows]), ref, "decode_gqa_fp8 sampled")

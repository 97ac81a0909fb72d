"""GPU parity of pa_prefill (tcgen05 tensor-core path) against the float64 oracle.

Tolerance for bf16 operands with fp32 accumulation and fp32 output:
max |err| <= 2e-3 and relative L2 <= 1e-3.  On the tensor cores Q K^T runs
on the bf16 operands and P V on fp16 operands (P and V rounded to fp16); the
oracle keeps everything in float64.  The V range tests check the documented
consequence: V values beyond the fp16 range are saturated and flagged,
values below its normal range keep an absolute error under 2^-25.
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


# --------------------------------------------------------------------------- V range
def _rescale_v(g, oc, picks, factor):
    """Replace the V rows of the (sequence, position) picks by factor x their
    value, rounded to bf16, in the device-resident KV pool (through pa_write_kv) and in the
    oracle's pool; K rows are rewritten unchanged."""
    Bp = g.wl.block_size
    gt = g.tables_list()
    slots = []
    for s, pos in picks:
        assert gt[s][pos // Bp] == oc.tables[s][pos // Bp]
        slots.append(oc.tables[s][pos // Bp] * Bp + pos % Bp)
    blk, off = np.asarray(slots) // Bp, np.asarray(slots) % Bp
    k_bits = np.ascontiguousarray(oc.k[blk, :, off, :])
    v_t = torch.from_numpy((oracle.bits_to_f64(oc.v[blk, :, off, :]) * factor)
                           .astype(np.float32)).to(torch.bfloat16)
    oracle.write_kv(oc.k, oc.v, k_bits, oracle.to_numpy_bits(v_t), slots)
    k_t = torch.from_numpy(k_bits.view(np.int16)).view(torch.bfloat16)
    pkv.write_kv(g.cache.pool, k_t.to(g.device), v_t.to(g.device),
                 torch.tensor(slots, dtype=torch.int64, device=g.device), d_err=g.err)


def _range_case():
    wl = workloads.custom_decode(3, 8, 2, 128, 16, "bf16", [100, 0, 257], seed=23,
                                 new_lens=[70, 129, 40], kind="prefill")
    g = GpuWorkload(wl)
    g.err.zero_()
    g.write_new()
    return wl, g, oracle.OracleCache(wl)


def _prefill_ref(wl, g, oc, kpool, vpool, q):
    cu = np.concatenate([[0], np.cumsum(wl.new_lens)])
    return oracle.prefill(kpool, vpool, q, cu, wl.total_lens, oc.tables, wl.scale,
                          causal=wl.causal)


def _fp16_pools(oc, q_bits):
    """The oracle's pools and queries as float64, V rounded to fp16 (to nearest
    even, saturating at +-65504): the values P V runs on."""
    v = np.clip(oracle.bits_to_f64(oc.v), -65504.0, 65504.0).astype(np.float16)
    return oracle.bits_to_f64(oc.k), v.astype(np.float64), oracle.bits_to_f64(q_bits)


def test_prefill_small_v_magnitudes():
    """V rows around 1e-6 (below the fp16 normal range): sequence 0 has every
    third key scaled, sequence 1 all of its keys.  Mixed rows meet the usual
    tolerance; all-small rows stay within 2^-25 (+ P rounding) of the exact
    result and within the relative tolerance of the fp16-rounded V."""
    wl, g, oc = _range_case()
    picks = [(0, p) for p in range(0, 170, 3)] + [(1, p) for p in range(129)]
    _rescale_v(g, oc, picks, 1e-6)
    g.attend()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0, pkv.status_str(int(g.err.item()))
    got = g.out.cpu().numpy().astype(np.float64)
    q = oracle.to_numpy_bits(g.q_host)
    ref = _prefill_ref(wl, g, oc, oc.k, oc.v, q)
    a, b = 70, 70 + 129  # query rows of sequence 1
    mixed = np.r_[0:a, b:got.shape[0]]
    _check(got[mixed], ref[mixed], "mixed small V")
    small, small_ref = got[a:b], ref[a:b]
    assert np.isfinite(small).all()
    assert np.abs(small_ref).max() > 1e-7  # the case really is small but not zero
    assert np.abs(small - small_ref).max() <= 2.0 ** -25 + 1e-3 * np.abs(small_ref).max()
    ref16 = _prefill_ref(wl, g, oc, *_fp16_pools(oc, q))[a:b]
    rel = np.linalg.norm(small - ref16) / np.linalg.norm(ref16)
    assert rel <= REL_L2, "all-small V vs fp16-rounded V: rel L2 %.3g" % rel


def test_prefill_v_beyond_fp16_range_is_flagged():
    """V rows around 1e5 in sequence 0: those values saturate at +-65504, the
    call sets PA_ERR_UNSUPPORTED, sequence 0's rows equal the attention over
    the saturated values and the other sequences are untouched."""
    wl, g, oc = _range_case()
    _rescale_v(g, oc, [(0, p) for p in range(0, 170, 7)], 1e5)
    assert np.abs(oracle.bits_to_f64(oc.v)[np.isfinite(oracle.bits_to_f64(oc.v))]).max() > 65504
    g.attend()
    torch.cuda.synchronize()
    assert int(g.err.item()) == pkv.PA_ERR_UNSUPPORTED
    got = g.out.cpu().numpy().astype(np.float64)
    q = oracle.to_numpy_bits(g.q_host)
    ref = _prefill_ref(wl, g, oc, oc.k, oc.v, q)
    _check(got[70:], ref[70:], "sequences without large V")
    sat = _prefill_ref(wl, g, oc, *_fp16_pools(oc, q))[:70]
    big = got[:70]
    assert np.isfinite(big).all()
    scale = np.abs(sat).max()
    rel = np.linalg.norm(big - sat) / np.linalg.norm(sat)
    assert rel <= REL_L2 and np.abs(big - sat).max() <= MAX_ABS * scale, (rel, scale)

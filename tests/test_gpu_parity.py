"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Inputs come from the seeded generators in workloads.py; the GPU side builds
its cache with the product allocator and pa_write_kv / pa_copy_blocks, the
oracle side with its own allocator and numpy writes.  Tolerances:
  - pa_write_kv, pa_copy_blocks, block tables: bit-exact;
  - bf16 attention (fp32 output): max |err| <= 2e-3 and relative L2 <= 1e-3;
  - fp32 attention: max |err| <= 1e-5.
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


def _pool_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def _oracle_bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint8).reshape(-1)


def assert_close(got, ref, dtype, what=""):
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), "%s: non-finite output" % what
    if dtype == "f32":
        assert err.max() <= F32_MAX_ABS, "%s max abs err %.3g" % (what, err.max())
    else:
        rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
        assert err.max() <= BF16_MAX_ABS, "%s max abs err %.3g" % (what, err.max())
        assert rel <= BF16_REL_L2, "%s rel L2 %.3g" % (what, rel)


def _run_both(wl, partition_tokens=0):
    g = GpuWorkload(wl)
    if partition_tokens:
        g.set_partition_tokens(partition_tokens)
    g.err.zero_()
    out = g.step()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0, pkv.status_str(int(g.err.item()))
    oc = oracle.OracleCache(wl)
    return g, oc, out.cpu().numpy()


# ---------------------------------------------------------------- write / copy / tables
WRITE_CASES = [
    ("tiny", lambda: workloads.decode_tiny()),
    ("gqa", lambda: workloads.decode_gqa(scale=1 / 8)),
    ("mha", lambda: workloads.decode_mha(scale=1 / 16)),
    ("long_shared", lambda: workloads.decode_long_shared(scale=1 / 256)),
    ("prefill", lambda: workloads.prefill(scale=1 / 8)),
]


@pytest.mark.parametrize("name,make", WRITE_CASES)
def test_write_kv_and_tables_bit_exact(name, make):
    wl = make()
    g = GpuWorkload(wl)
    g.err.zero_()
    g.write_new()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    oc = oracle.OracleCache(wl)
    assert g.tables_list() == oc.tables
    assert g.cow_pairs == oc.cow_pairs
    assert np.array_equal(_pool_bits(g.cache.pool.k).reshape(-1), _oracle_bits(oc.k))
    assert np.array_equal(_pool_bits(g.cache.pool.v).reshape(-1), _oracle_bits(oc.v))


def test_write_kv_rejects_out_of_pool_slot_and_writes_the_rest():
    wl = workloads.decode_gqa(scale=1 / 8)
    g = GpuWorkload(wl)
    assert wl.num_seqs >= 4
    before_k = _pool_bits(g.cache.pool.k).copy()
    bad = g.slot_mapping.clone()
    n_slots = wl.num_blocks * wl.block_size
    bad[0] = n_slots            # one past the pool
    bad[1] = -5
    g.err.zero_()
    pkv.write_kv(g.cache.pool, g.k_new, g.v_new, bad, d_err=g.err)
    torch.cuda.synchronize()
    assert int(g.err.item()) == pkv.PA_ERR_OUT_OF_RANGE
    after_k = _pool_bits(g.cache.pool.k)
    # rows 2.. were written, rows 0/1 skipped
    oc = oracle.OracleCache(wl, write_new=False)
    ok_slots = g.slot_mapping_host[2:]
    oracle.write_kv(oc.k, oc.v, oracle.to_numpy_bits(g.k_new_host[2:]),
                    oracle.to_numpy_bits(g.v_new_host[2:]), ok_slots)
    assert np.array_equal(after_k.reshape(-1), _oracle_bits(oc.k))
    assert not np.array_equal(before_k, after_k)


@pytest.mark.parametrize("block_size,dtype,D", [(16, "bf16", 128), (4, "f32", 64), (1, "bf16", 64)])
def test_copy_blocks_bit_exact(block_size, dtype, D):
    wl = workloads.custom_decode(6, 8, 2, D, block_size, dtype, [37, 5, 64, 1, 90, 17], seed=3)
    g = GpuWorkload(wl)
    g.write_new()
    oc = oracle.OracleCache(wl)
    rng = np.random.default_rng(4)
    held = sorted({b for t in oc.tables for b in t})
    free = sorted(set(range(wl.num_blocks)) - set(held))
    n = min(len(held), len(free), 9)
    src = rng.choice(held, n, replace=False).astype(np.int32)
    dst = rng.choice(free, n, replace=False).astype(np.int32)
    g.err.zero_()
    pkv.copy_blocks(g.cache.pool, torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda(),
                    d_err=g.err)
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    oracle.copy_blocks(oc.k, oc.v, src.tolist(), dst.tolist())
    assert np.array_equal(_pool_bits(g.cache.pool.k).reshape(-1), _oracle_bits(oc.k))
    assert np.array_equal(_pool_bits(g.cache.pool.v).reshape(-1), _oracle_bits(oc.v))
    # an id outside the pool is flagged and skipped
    g.err.zero_()
    pkv.copy_blocks(g.cache.pool, torch.tensor([0], dtype=torch.int32, device="cuda"),
                    torch.tensor([wl.num_blocks], dtype=torch.int32, device="cuda"), d_err=g.err)
    torch.cuda.synchronize()
    assert int(g.err.item()) == pkv.PA_ERR_OUT_OF_RANGE


# ---------------------------------------------------------------- decode parity
DECODE_CASES = [
    ("tiny", lambda: workloads.decode_tiny()),
    ("gqa_small", lambda: workloads.decode_gqa(scale=1 / 8)),
    ("mha_small", lambda: workloads.decode_mha(scale=1 / 8)),
    ("long_shared_small", lambda: workloads.decode_long_shared(scale=1 / 64)),
]


@pytest.mark.parametrize("name,make", DECODE_CASES)
def test_decode_matches_oracle(name, make):
    wl = make()
    g, oc, got = _run_both(wl)
    ref = oracle.decode(oc.k, oc.v, oracle.to_numpy_bits(g.q_host), oc.tables, wl.total_lens,
                        wl.scale)
    assert_close(got, ref, wl.dtype, name)


@pytest.mark.parametrize("part", [16, 32, 48, 256, 1 << 20])
def test_decode_partition_sizes(part):
    # many partitions (merge kernel), uneven ones, and a single partition
    wl = workloads.decode_gqa(scale=1 / 16)
    g, oc, got = _run_both(wl, partition_tokens=part)
    ref = oracle.decode(oc.k, oc.v, oracle.to_numpy_bits(g.q_host), oc.tables, wl.total_lens,
                        wl.scale)
    assert_close(got, ref, wl.dtype, "part=%d" % part)


EDGE_LENS = [0, 1, 14, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 129, 300]


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("block_size", [1, 2, 4, 8, 16, 32, 64])
def test_decode_edge_lengths_bf16(G, block_size):
    # cached lengths around chunk (16) and block boundaries; new token makes n = c + 1
    wl = workloads.custom_decode(len(EDGE_LENS), 2 * G, 2, 128, block_size, "bf16", EDGE_LENS,
                                 seed=G * 100 + block_size)
    for part in (0, 32):
        g, oc, got = _run_both(wl, partition_tokens=part)
        ref = oracle.decode(oc.k, oc.v, oracle.to_numpy_bits(g.q_host), oc.tables, wl.total_lens,
                            wl.scale)
        assert_close(got, ref, "bf16", "G=%d bp=%d part=%d" % (G, block_size, part))


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("block_size", [1, 4, 16])
def test_decode_edge_lengths_f32(G, block_size):
    wl = workloads.custom_decode(len(EDGE_LENS), 2 * G, 2, 64, block_size, "f32", EDGE_LENS,
                                 seed=G * 10 + block_size)
    g, oc, got = _run_both(wl, partition_tokens=48)
    ref = oracle.decode(oc.k, oc.v, oracle.to_numpy_bits(g.q_host), oc.tables, wl.total_lens,
                        wl.scale)
    assert_close(got, ref, "f32", "G=%d bp=%d" % (G, block_size))


def test_decode_result_does_not_depend_on_placement():
    # the same logical content under two physical placements gives identical bits
    wl = workloads.decode_gqa(scale=1 / 16)
    a = GpuWorkload(wl)
    out_a = a.step().clone()
    wl2 = workloads.decode_gqa(scale=1 / 16)
    wl2.free_order = np.random.default_rng(77).permutation(wl2.num_blocks).astype(np.int32)
    b = GpuWorkload(wl2)
    out_b = b.step()
    torch.cuda.synchronize()
    assert a.tables_list() != b.tables_list()
    assert torch.equal(out_a, out_b)


def test_decode_flags_table_entry_outside_pool():
    wl = workloads.decode_gqa(scale=1 / 32)
    g = GpuWorkload(wl)
    g.write_new()
    bt = g.block_tables.clone()
    bt[0, 0] = wl.num_blocks + 3
    bt[1, 0] = -2
    g.err.zero_()
    pkv.decode(g.cache.pool, g.q, bt, g.context_lens, g.max_context, wl.scale, out=g.out,
               workspace=g.workspace, d_err=g.err)
    torch.cuda.synchronize()
    assert int(g.err.item()) in (pkv.PA_ERR_OUT_OF_RANGE, pkv.PA_ERR_NEGATIVE_BLOCK)


def test_decode_clamps_contexts_above_max_context():
    # a context longer than max_context is cut to its first max_context
    # positions and flagged; the other sequences are unaffected
    wl = workloads.decode_gqa(scale=1 / 8)
    g = GpuWorkload(wl)
    g.write_new()
    n = wl.total_lens.astype(np.int64)
    cap = int(n.max()) - 5
    assert cap >= 1 and int((n > cap).sum()) >= 1
    g.err.zero_()
    out = pkv.decode(g.cache.pool, g.q, g.block_tables, g.context_lens, cap, wl.scale, d_err=g.err)
    torch.cuda.synchronize()
    assert int(g.err.item()) == pkv.PA_ERR_OUT_OF_RANGE
    oc = oracle.OracleCache(wl)
    ref = oracle.decode(oc.k, oc.v, oracle.to_numpy_bits(g.q_host), oc.tables,
                        np.minimum(n, cap), wl.scale)
    assert_close(out.cpu().numpy(), ref, "bf16", "max_context=%d" % cap)


# ---------------------------------------------------------------- full-size workloads
@pytest.mark.parametrize("make", [workloads.decode_tiny, workloads.decode_gqa,
                                  workloads.decode_mha, workloads.decode_long_shared],
                         ids=["decode_tiny", "decode_gqa", "decode_mha", "decode_long_shared"])
def test_decode_full_size_matches_oracle(make):
    wl = make()
    g, oc, got = _run_both(wl)
    q = oracle.to_numpy_bits(g.q_host)
    if wl.num_seqs * wl.num_q_heads * float(wl.total_lens.mean()) <= 8e7:
        ref = oracle.decode(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale)
        assert_close(got, ref, wl.dtype, wl.name)
    else:
        rng = np.random.default_rng(9)
        rows = [(int(s), int(h)) for s, h in zip(rng.integers(0, wl.num_seqs, 96),
                                                 rng.integers(0, wl.num_q_heads, 96))]
        ref = oracle.decode(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale, rows=rows)
        sel = np.stack([got[s, h] for s, h in rows])
        assert_close(sel, ref, wl.dtype, wl.name + " sampled")

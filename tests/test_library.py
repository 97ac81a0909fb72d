"""Host-side checks of libpagedkv.so (no GPU needed).

The library must build for sm_103a, load, and export every symbol the C
header declares.  Its host functions (slot arithmetic, allocator) are checked
against the pages' worked examples and against the oracle's independent
allocator on random operation sequences.  Argument errors that are caught on
the host return their status without touching a device.
"""
import ctypes
import json
import os
import random
import re

import numpy as np
import pytest

import oracle
import paged_kv_cache_148_gb300 as pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def L():
    pkv.build()
    return pkv.lib()


def _declared_symbols():
    with open(os.path.join(ROOT, "include", "pagedkv.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    declared = _declared_symbols()
    assert len(declared) >= 20
    missing = [s for s in declared if not hasattr(L, s)]
    assert not missing, missing
    assert sorted(pkv.EXPORTED) == declared


def test_library_is_built_for_sm_103a():
    from paged_kv_cache_148_gb300 import builder
    assert "arch=compute_103a,code=sm_103a" in builder.ARCH
    assert builder.up_to_date()


def test_status_strings(L):
    for code in range(9):
        assert pkv.status_str(code).startswith("PA_")
    assert L.pa_abi_version() == 2


def test_physical_slot_worked_example(L):
    with open(os.path.join(GOLDEN, "physical_slot_example.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        assert pkv.physical_slot(g["block_table"], g["block_size"], case["pos"]) == case["slot"]
    expect = {"IndexError": pkv.PA_ERR_OUT_OF_RANGE, "ValueError": None}
    for case in g["failures"]:
        with pytest.raises(pkv.PagedKVError) as ei:
            pkv.physical_slot(case["block_table"], case["block_size"], case["pos"])
        if case["error"] == "IndexError":
            assert ei.value.status == pkv.PA_ERR_OUT_OF_RANGE
        else:
            assert ei.value.status in (pkv.PA_ERR_INVALID_ARG, pkv.PA_ERR_NEGATIVE_BLOCK)


def test_slot_mapping_matches_oracle(L):
    rng = np.random.default_rng(0)
    for bp in (1, 3, 4, 16, 64):
        table = rng.permutation(500)[:20].tolist()
        pos = rng.integers(0, 20 * bp, size=300)
        got = pkv.slot_mapping(table, bp, pos)
        ref = [oracle.physical_slot(table, bp, int(p)) for p in pos]
        assert got.tolist() == ref


def test_page_size_bytes(L):
    pool = pkv.pa_kv_pool(1, 1, 10, 16, 2, 128, pkv.DTYPE_BF16)
    out = ctypes.c_int64()
    assert L.pa_page_size_bytes(ctypes.byref(pool), ctypes.byref(out)) == 0
    assert out.value == 2 * 16 * 2 * 128 * 2
    pool.dtype = 7
    assert L.pa_page_size_bytes(ctypes.byref(pool), ctypes.byref(out)) == pkv.PA_ERR_INVALID_ARG


def test_cow_worked_example_on_product_allocator(L):
    with open(os.path.join(GOLDEN, "cow_example.json")) as f:
        g = json.load(f)
    # the example's state: parent [7] (refcount 1) and 9 next on the free list
    n = g["num_blocks"]
    a = pkv.Allocator(n, [b for b in range(n) if b not in (7, 9)] + [9, 7])
    parent = pkv.BlockTable()
    assert a.append(parent) == 7
    child = a.fork(parent)
    blk, off, cow = a.writable_tail(child, g["logical_length"], g["block_size"])
    e = g["expect"]
    assert (blk, off, cow) == (e["block"], e["offset"], e["cow_src"])
    assert parent.tolist() == e["parent_after"] and child.tolist() == e["child_after"]
    for b, r in e["refcount_after"].items():
        assert a.refcount(int(b)) == r


def test_allocator_matches_oracle_on_random_sequences(L):
    rng = random.Random(5)
    for trial in range(40):
        n_blocks = 48
        bp = rng.choice([1, 2, 4, 16])
        order = rng.sample(range(n_blocks), n_blocks)
        ref = oracle.BlockPool(n_blocks, order)
        got = pkv.Allocator(n_blocks, order)
        rt, gt, lens = [], [], []
        for step in range(150):
            op = rng.random()
            if op < 0.15 or not rt:
                rt.append([]), gt.append(pkv.BlockTable()), lens.append(0)
            elif op < 0.3:
                i = rng.randrange(len(rt))
                rt.append(ref.fork(rt[i]))
                gt.append(got.fork(gt[i]))
                lens.append(lens[i])
            elif op < 0.85:
                i = rng.randrange(len(rt))
                try:
                    r = ref.writable_tail(rt[i], lens[i], bp)
                except MemoryError:
                    with pytest.raises(pkv.PagedKVError) as ei:
                        got.writable_tail(gt[i], lens[i], bp)
                    assert ei.value.status == pkv.PA_ERR_NO_FREE_BLOCK
                    break
                g = got.writable_tail(gt[i], lens[i], bp)
                assert r == g
                lens[i] += 1
            else:
                i = rng.randrange(len(rt))
                ref.release(rt[i])
                got.release(gt[i])
                rt.pop(i), gt.pop(i), lens.pop(i)
            assert [t for t in rt] == [t.tolist() for t in gt]
            assert ref.refcount == [got.refcount(b) for b in range(n_blocks)]
            assert len(ref.free) == got.num_free()


def test_reserve_equals_repeated_writable_tail(L):
    order = list(range(200))
    random.Random(1).shuffle(order)
    a = pkv.Allocator(200, order)
    b = oracle.BlockPool(200, order)
    ta, tb = pkv.BlockTable(), []
    slots, cows = a.reserve(ta, 0, 37, 4)
    ref_slots = []
    for pos in range(37):
        blk, off, _ = b.writable_tail(tb, pos, 4)
        ref_slots.append(blk * 4 + off)
    assert slots.tolist() == ref_slots and cows == []
    child_a, child_b = a.fork(ta), b.fork(tb)
    s2, cows = a.reserve(child_a, 37, 5, 4)
    ref = [b.writable_tail(child_b, 37 + i, 4) for i in range(5)]
    assert s2.tolist() == [x[0] * 4 + x[1] for x in ref]
    assert cows == [(x[2], x[0]) for x in ref if x[2] >= 0] and len(cows) == 1


def test_allocator_errors(L):
    a = pkv.Allocator(2)
    t = pkv.BlockTable()
    a.append(t)
    a.append(t)
    with pytest.raises(pkv.PagedKVError) as ei:
        a.append(t)
    assert ei.value.status == pkv.PA_ERR_NO_FREE_BLOCK
    stale = pkv.BlockTable(ids=t.tolist())
    a.release(t)
    with pytest.raises(pkv.PagedKVError) as ei:
        a.release(stale)
    assert ei.value.status == pkv.PA_ERR_REFCOUNT
    with pytest.raises(pkv.PagedKVError) as ei:
        a.writable_tail(pkv.BlockTable(), 5, 4)   # logical block 1 not allocated
    assert ei.value.status == pkv.PA_ERR_OUT_OF_RANGE
    with pytest.raises(pkv.PagedKVError):
        pkv.Allocator(3, [0, 0, 1])               # not a permutation


def test_new_block_only_at_the_end_of_the_table(L):
    # a block boundary inside the table or past its end is not the next
    # block: INVALID_ARG, with the table and the refcounts unchanged (the
    # oracle's BlockPool rejects the same calls)
    a = pkv.Allocator(8)
    t = pkv.BlockTable()
    for length in (0, 4):
        a.writable_tail(t, length, 4)
    before = (t.tolist(), [a.refcount(b) for b in range(8)])
    for length in (4, 16):
        with pytest.raises(pkv.PagedKVError) as ei:
            a.writable_tail(t, length, 4)
        assert ei.value.status == pkv.PA_ERR_INVALID_ARG
    assert (t.tolist(), [a.refcount(b) for b in range(8)]) == before


def test_device_entry_points_reject_bad_arguments_on_host(L):
    # these return before any CUDA call, so they run without a GPU
    P = ctypes.c_void_p
    null_pool = None
    assert L.pa_write_kv(null_pool, P(16), P(16), P(16), 1, None, None) == pkv.PA_ERR_INVALID_ARG
    pool = pkv.pa_kv_pool(16, 16, 10, 16, 8, 128, pkv.DTYPE_BF16)
    pp = ctypes.byref(pool)
    assert L.pa_write_kv(pp, P(16), P(16), P(16), -1, None, None) == pkv.PA_ERR_INVALID_ARG
    assert L.pa_write_kv(pp, P(16), P(16), P(16), 0, None, None) == pkv.PA_OK
    assert L.pa_copy_blocks(pp, P(16), P(16), 0, None, None) == pkv.PA_OK
    assert L.pa_copy_blocks(pp, None, P(16), 3, None, None) == pkv.PA_ERR_INVALID_ARG
    # decode: head groups that do not divide, an unsupported head_dim
    args = [P(16), 30, P(16), 4, P(16), 2, 64, ctypes.c_float(0.1), 0, P(16), None, 0, None, None]
    assert L.pa_decode(pp, *args) == pkv.PA_ERR_INVALID_ARG
    pool.head_dim = 96
    args[1] = 32
    assert L.pa_decode(pp, *args) == pkv.PA_ERR_UNSUPPORTED
    pool.head_dim = 128
    pool.block_size = 12
    assert L.pa_decode(pp, *args) == pkv.PA_ERR_UNSUPPORTED
    pool.block_size = 16
    args[8] = 17   # partition not a multiple of 16
    assert L.pa_decode(pp, *args) == pkv.PA_ERR_INVALID_ARG


def test_workspace_sizes(L):
    pool = pkv.pa_kv_pool(16, 16, 10, 16, 8, 128, pkv.DTYPE_BF16)
    pp = ctypes.byref(pool)
    out = ctypes.c_size_t()
    # one partition covers everything -> no workspace
    assert L.pa_decode_workspace_bytes(pp, 4, 32, 100, 4096, ctypes.byref(out)) == 0
    assert out.value == 0
    # 64-token partitions over 1000 tokens -> 16 partitions of (D + 2) floats each
    assert L.pa_decode_workspace_bytes(pp, 4, 32, 1000, 64, ctypes.byref(out)) == 0
    rows = 4 * 32 * 16
    assert out.value >= rows * (128 + 2) * 4
    pt = ctypes.c_int32()
    assert L.pa_decode_partition_tokens(pp, 64, 32, 4097, ctypes.byref(pt)) == 0
    assert pt.value > 0 and pt.value % 16 == 0


def test_fp8_pool_page_size_and_argument_checks(L):
    # FP8 pages count one byte per element plus a float32 scale per row
    pool = pkv.pa_kv_pool(1, 1, 10, 16, 2, 128, pkv.DTYPE_FP8_E4M3, 16, 16)
    out = ctypes.c_int64()
    assert L.pa_page_size_bytes(ctypes.byref(pool), ctypes.byref(out)) == 0
    assert out.value == 2 * 16 * 2 * (128 + 4)
    P = ctypes.c_void_p
    pp = ctypes.byref(pool)
    # the scale arrays are required
    nos = pkv.pa_kv_pool(16, 16, 10, 16, 2, 128, pkv.DTYPE_FP8_E4M3, None, None)
    assert L.pa_write_kv(ctypes.byref(nos), P(16), P(16), P(16), 1, None, None) == \
        pkv.PA_ERR_INVALID_ARG
    # only D = 128 rows are written; decode needs blocks of at least 4 tokens
    pool.head_dim = 64
    assert L.pa_write_kv(pp, P(16), P(16), P(16), 1, None, None) == pkv.PA_ERR_UNSUPPORTED
    pool.head_dim = 128
    pool.block_size = 2
    args = [P(16), 4, P(16), 4, P(16), 2, 64, ctypes.c_float(0.1), 0, P(16), None, 0, None, None]
    assert L.pa_decode(pp, *args) == pkv.PA_ERR_UNSUPPORTED
    # the one-launch step writes raw rows and so takes no FP8 pool
    pool.block_size = 16
    step = [P(16), P(16), P(16), P(16), 4, P(16), 4, P(16), 2, 64, ctypes.c_float(0.1), 0,
            P(16), None, 0, None, None]
    assert L.pa_decode_step(pp, *step) == pkv.PA_ERR_UNSUPPORTED
    # a window must be positive
    win = [P(16), 4, P(16), 4, P(16), 2, 64, 0, ctypes.c_float(0.1), 0, P(16), None, 0, None,
           None]
    pool.dtype = pkv.DTYPE_BF16
    assert L.pa_decode_window(pp, *win) == pkv.PA_ERR_INVALID_ARG


def test_plan_properties_over_random_shapes(L):
    # the automatic partition size is a whole number of 4-warp rounds of
    # 16-token chunks, and every workspace holds (max, sum, D values) for each
    # (sequence, q-head, partition); a window never needs more than the whole
    # context
    rng = np.random.default_rng(23)
    for _ in range(300):
        Hkv = int(rng.choice([1, 2, 4, 8, 16]))
        G = int(rng.choice([1, 2, 4, 8]))
        B = int(rng.integers(1, 300))
        max_ctx = int(rng.integers(1, 300000))
        pool = pkv.pa_kv_pool(16, 16, 1000, 16, Hkv, 128, pkv.DTYPE_BF16)
        pp = ctypes.byref(pool)
        pt = ctypes.c_int32()
        assert L.pa_decode_partition_tokens(pp, B, G * Hkv, max_ctx, ctypes.byref(pt)) == 0
        assert pt.value >= 128 and pt.value % 64 == 0
        out = ctypes.c_size_t()
        assert L.pa_decode_workspace_bytes(pp, B, G * Hkv, max_ctx, 0, ctypes.byref(out)) == 0
        parts = -(-(-(-max_ctx // 16)) // (pt.value // 16))
        if parts > 1:
            assert out.value >= B * G * Hkv * parts * (128 + 2) * 4
        else:
            assert out.value == 0
        w = int(rng.integers(1, 5000))
        wout = ctypes.c_size_t()
        assert L.pa_decode_window_workspace_bytes(pp, B, G * Hkv, max_ctx, w, 0,
                                                  ctypes.byref(wout)) == 0
        if w >= max_ctx:
            assert wout.value <= out.value

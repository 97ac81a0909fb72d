"""Pins of the float64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: values the
pages print (tests/golden/), a library softmax-attention routine, closed
forms, invariants the pages state, or an identity that must hold exactly.
"""
import json
import math
import os
import random

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------- addressing (worked example)
@pytest.mark.parametrize("impl", [oracle.physical_slot, oracle.physical_slot_c])
def test_physical_slot_worked_example(impl):
    g = _golden("physical_slot_example.json")
    for case in g["cases"]:
        assert impl(g["block_table"], g["block_size"], case["pos"]) == case["slot"]


@pytest.mark.parametrize("impl", [oracle.physical_slot, oracle.physical_slot_c])
def test_physical_slot_failures(impl):
    g = _golden("physical_slot_example.json")
    for case in g["failures"]:
        exc = {"IndexError": IndexError, "ValueError": ValueError}[case["error"]]
        with pytest.raises(exc):
            impl(case["block_table"], case["block_size"], case["pos"])


def test_physical_slot_lands_on_table_block_same_offset():
    # invariant of P2 "Page-table 寻址": each allocated position lands in the
    # table's block at the same in-block offset, and nothing past the table.
    rng = random.Random(3)
    for _ in range(200):
        bp = rng.choice([1, 2, 3, 4, 5, 16, 32])
        table = rng.sample(range(1000), rng.randint(1, 9))
        for pos in range(len(table) * bp):
            slot = oracle.physical_slot(table, bp, pos)
            assert slot // bp == table[pos // bp]
            assert slot % bp == pos % bp
        with pytest.raises(IndexError):
            oracle.physical_slot(table, bp, len(table) * bp)


# ----------------------------------------------------------------- ownership (worked example)
def test_fork_and_writable_tail_worked_example():
    g = _golden("cow_example.json")
    pool = oracle.BlockPool(g["num_blocks"], free_order=g["free"])
    for b, r in g["refcount"].items():
        pool.refcount[int(b)] = r
    parent = list(g["parent"])
    child = pool.fork(parent)
    block, offset, cow = pool.writable_tail(child, g["logical_length"], g["block_size"])
    e = g["expect"]
    assert (block, offset) == (e["block"], e["offset"])
    assert parent == e["parent_after"] and child == e["child_after"]
    assert {int(k): pool.refcount[int(k)] for k in e["refcount_after"]} == \
        {int(k): v for k, v in e["refcount_after"].items()}
    assert cow == e["cow_src"]


def _holders(tables, b):
    return sum(t.count(b) for t in tables)


def test_refcount_and_cow_invariants_random_sequences():
    # P2 "生命周期与所有权": refcount == number of holding sequences; a shared
    # block is never written in place; free and held blocks are disjoint.
    rng = random.Random(11)
    for trial in range(60):
        n_blocks = 64
        bp = rng.choice([2, 4, 16])
        pool = oracle.BlockPool(n_blocks, rng.sample(range(n_blocks), n_blocks))
        tables, lengths = [], []
        for step in range(120):
            op = rng.random()
            try:
                if op < 0.15 or not tables:
                    tables.append([])
                    lengths.append(0)
                elif op < 0.30:
                    i = rng.randrange(len(tables))
                    tables.append(pool.fork(tables[i]))
                    lengths.append(lengths[i])
                elif op < 0.85:
                    i = rng.randrange(len(tables))
                    blk, off, cow = pool.writable_tail(tables[i], lengths[i], bp)
                    # the block written to is exclusively owned
                    assert pool.refcount[blk] == 1
                    assert _holders(tables, blk) == 1
                    assert off == lengths[i] % bp
                    if cow >= 0:
                        assert off != 0 and cow != blk
                    lengths[i] += 1
                else:
                    i = rng.randrange(len(tables))
                    pool.release(tables[i])
                    tables.pop(i)
                    lengths.pop(i)
            except MemoryError:
                break
            for b in range(n_blocks):
                assert pool.refcount[b] == _holders(tables, b)
            assert len(set(pool.free)) == len(pool.free)
            held = {b for t in tables for b in t}
            assert held.isdisjoint(pool.free)
            assert len(held) + len(pool.free) == n_blocks


def test_new_block_only_at_the_end_of_the_table():
    # position len(table) * B_p starts the next logical block; a position at a
    # block boundary inside the table names a block that is already mapped,
    # so appending there would break "one physical block per logical block"
    pool = oracle.BlockPool(8)
    table = []
    for length in (0, 4):
        pool.writable_tail(table, length, 4)
    before = (list(table), list(pool.refcount), list(pool.free))
    with pytest.raises(ValueError):
        pool.writable_tail(table, 4, 4)
    with pytest.raises(ValueError):
        pool.writable_tail(table, 16, 4)
    assert (table, pool.refcount, pool.free) == before


def test_release_underflow_is_an_error():
    pool = oracle.BlockPool(4)
    t = []
    pool.append(t)
    stale = list(t)
    pool.release(t)
    with pytest.raises(ValueError):
        pool.release(stale)


def test_pool_exhaustion_is_an_error():
    pool = oracle.BlockPool(2)
    t = []
    pool.append(t)
    pool.append(t)
    with pytest.raises(MemoryError):
        pool.append(t)


# ----------------------------------------------------------------- attention
def _small_case(dtype, G, Hkv, D, bp, lens, seed):
    wl = workloads.custom_decode(len(lens), G * Hkv, Hkv, D, bp, dtype,
                                 [n - 1 for n in lens], seed=seed)
    oc = oracle.OracleCache(wl)
    q = oracle.to_numpy_bits(wl.queries())
    return wl, oc, q


def _gathered(oc, s, n):
    """Logical K/V of sequence s (float64 [n][H][D]) read through its table."""
    bp = oc.wl.block_size
    k = np.stack([oracle.bits_to_f64(oc.k[oc.tables[s][i // bp], :, i % bp]) for i in range(n)])
    v = np.stack([oracle.bits_to_f64(oc.v[oc.tables[s][i // bp], :, i % bp]) for i in range(n)])
    return k, v


CASES = [
    ("f32", 1, 2, 64, 4, [1, 4, 5, 17]),
    ("f32", 2, 2, 64, 4, [3, 64, 65]),
    ("bf16", 4, 2, 128, 16, [1, 16, 17, 40]),
    ("bf16", 8, 1, 128, 16, [33, 2]),
    ("bf16", 2, 3, 32, 1, [7, 9]),
    ("f32", 3, 2, 16, 5, [11, 26]),
]


@pytest.mark.parametrize("dtype,G,Hkv,D,bp,lens", CASES)
def test_decode_matches_library_sdpa(dtype, G, Hkv, D, bp, lens):
    wl, oc, q = _small_case(dtype, G, Hkv, D, bp, lens, seed=len(lens) + D)
    got = oracle.decode(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale)
    qf = oracle.bits_to_f64(q)
    for s, n in enumerate(wl.total_lens):
        k, v = _gathered(oc, s, int(n))
        for g in range(wl.num_q_heads):
            h = g // G
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(qf[s, g][None, None, None]),
                torch.from_numpy(k[:, h][None, None]),
                torch.from_numpy(v[:, h][None, None]), scale=wl.scale)[0, 0, 0].numpy()
            np.testing.assert_allclose(got[s, g], ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("dtype,G,Hkv,D,bp,lens", CASES[:3])
def test_decode_matches_numpy_softmax(dtype, G, Hkv, D, bp, lens):
    wl, oc, q = _small_case(dtype, G, Hkv, D, bp, lens, seed=99)
    got = oracle.decode(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale)
    qf = oracle.bits_to_f64(q)
    for s, n in enumerate(wl.total_lens):
        k, v = _gathered(oc, s, int(n))
        for g in range(wl.num_q_heads):
            logits = wl.scale * (k[:, g // G] @ qf[s, g])
            w = np.exp(logits - logits.max())
            ref = (w[:, None] * v[:, g // G]).sum(0) / w.sum()
            np.testing.assert_allclose(got[s, g], ref, rtol=1e-12, atol=1e-13)


def test_single_key_returns_its_value_exactly():
    wl, oc, q = _small_case("bf16", 4, 2, 128, 16, [1, 1, 1], seed=5)
    got = oracle.decode(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale)
    for s in range(3):
        for g in range(8):
            v0 = oracle.bits_to_f64(oc.v[oc.tables[s][0], g // 4, 0])
            assert np.array_equal(got[s, g], v0)


def test_identical_keys_give_mean_of_values():
    wl, oc, q = _small_case("f32", 2, 2, 64, 4, [13, 30], seed=6)
    for s in range(2):
        n = int(wl.total_lens[s])
        k0 = oc.k[oc.tables[s][0], :, 0].copy()
        for i in range(n):
            oc.k[oc.tables[s][i // 4], :, i % 4] = k0
    got = oracle.decode(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale)
    for s in range(2):
        _, v = _gathered(oc, s, int(wl.total_lens[s]))
        for g in range(4):
            np.testing.assert_allclose(got[s, g], v[:, g // 2].mean(0), rtol=1e-13, atol=1e-14)


def test_dominant_key_selects_its_value():
    wl, oc, q = _small_case("f32", 1, 1, 16, 4, [9], seed=8)
    q = np.ones_like(q)
    oc.k[oc.tables[0][1], 0, 2] = 1e4      # position 6 dominates every other logit
    got = oracle.decode(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale)
    np.testing.assert_allclose(got[0, 0], oc.v[oc.tables[0][1], 0, 2], rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype,G,Hkv,D,bp,lens", CASES)
def test_paged_equals_contiguous_bit_for_bit(dtype, G, Hkv, D, bp, lens):
    # P1 §4 / P3 §五: paging changes addressing, not the result.
    wl, oc, q = _small_case(dtype, G, Hkv, D, bp, lens, seed=21)
    paged = oracle.decode(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale)
    max_seq = int(max(wl.total_lens))
    kc = np.zeros((wl.num_seqs, max_seq, Hkv, D), oc.k.dtype)
    vc = np.zeros_like(kc)
    for s in range(wl.num_seqs):
        for i in range(int(wl.total_lens[s])):
            kc[s, i] = oc.k[oc.tables[s][i // bp], :, i % bp]
            vc[s, i] = oc.v[oc.tables[s][i // bp], :, i % bp]
    contig = oracle.decode_contiguous(kc, vc, q, wl.total_lens, wl.scale)
    assert np.array_equal(paged, contig)


def test_placement_does_not_change_the_result():
    # the same logical content under two different physical placements
    wl, oc, q = _small_case("bf16", 4, 2, 128, 16, [40, 70, 16], seed=31)
    a = oracle.decode(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale)
    perm = np.random.default_rng(0).permutation(wl.num_blocks)
    k2, v2 = np.empty_like(oc.k), np.empty_like(oc.v)
    k2[perm] = oc.k
    v2[perm] = oc.v
    tables2 = [[int(perm[b]) for b in t] for t in oc.tables]
    b = oracle.decode(k2, v2, q, tables2, wl.total_lens, wl.scale)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("part", [1, 3, 16, 17, 64, 1000])
def test_split_merge_equals_unsplit(part):
    # P1 §4: (max, exp_sum, weighted_value) states merge to the full result.
    wl, oc, q = _small_case("bf16", 4, 2, 128, 16, [1, 17, 100, 250], seed=41)
    full = oracle.decode(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale)
    split = oracle.decode_split(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale, part)
    np.testing.assert_allclose(split, full, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("first", [True, False])
def test_split_merge_with_far_apart_partition_maxima(first):
    # one key scores 1000 above the rest: every partition state must be taken
    # relative to the largest partition max (e^1000 overflows a double), and
    # the result is that key's value (the dominant-key closed form)
    n, D, bp = 12, 4, 4
    k = np.zeros((3, 1, bp, D))
    v = np.arange(3 * bp * D, dtype=np.float64).reshape(3, 1, bp, D) / 7.0
    k[:, 0, :, 1] = np.linspace(-1.0, 1.0, n).reshape(3, bp)
    hot = 0 if first else n - 1
    k[hot // bp, 0, hot % bp, 0] = 1000.0
    q = np.array([[[1.0, 1.0, 0.0, 0.0]]])
    tables, lens = [[0, 1, 2]], [n]
    full = oracle.decode(k, v, q, tables, lens, 1.0)
    split = oracle.decode_split(k, v, q, tables, lens, 1.0, bp)
    assert np.isfinite(split).all()
    assert np.array_equal(full[0, 0], v[hot // bp, 0, hot % bp])
    assert np.array_equal(split[0, 0], v[hot // bp, 0, hot % bp])


def test_gqa_head_mapping():
    # q-head g reads kv-head g // G: changing kv-head 1 changes only heads 4..7
    wl, oc, q = _small_case("bf16", 4, 2, 128, 16, [30, 50], seed=51)
    a = oracle.decode(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale)
    oc.v[:, 1] = oc.v[:, 0]
    oc.k[:, 1] = oc.k[:, 0]
    b = oracle.decode(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale)
    assert np.array_equal(a[:, :4], b[:, :4])
    assert not np.allclose(a[:, 4:], b[:, 4:])
    # and with kv-head 1 == kv-head 0 and equal queries, heads 0 and 4 agree
    q2 = q.copy()
    q2[:, 4] = q2[:, 0]
    c = oracle.decode(oc.k, oc.v, q2, oc.tables, wl.total_lens, wl.scale)
    assert np.array_equal(c[:, 0], c[:, 4])


def test_decode_out_of_range_table_fails():
    wl, oc, q = _small_case("f32", 2, 2, 64, 4, [9], seed=61)
    with pytest.raises(IndexError):
        oracle.decode(oc.k, oc.v, q, [oc.tables[0][:1]], wl.total_lens, wl.scale)


# ----------------------------------------------------------------- prefill
def _prefill_case(cached, new, seed, causal=True, dtype="bf16", G=4, Hkv=2, D=128, bp=16):
    wl = workloads.custom_decode(len(cached), G * Hkv, Hkv, D, bp, dtype, cached, seed=seed,
                                 new_lens=new, kind="prefill", causal=causal)
    oc = oracle.OracleCache(wl)
    q = oracle.to_numpy_bits(wl.queries())
    cu = np.concatenate([[0], np.cumsum(wl.new_lens)]).astype(np.int32)
    return wl, oc, q, cu


def test_prefill_causal_row_equals_truncated_decode():
    wl, oc, q, cu = _prefill_case([20, 0, 33], [12, 5, 17], seed=71)
    got = oracle.prefill(oc.k, oc.v, q, cu, wl.total_lens, oc.tables, wl.scale, causal=True)
    for s in range(wl.num_seqs):
        for i in range(int(wl.new_lens[s])):
            t = cu[s] + i
            n_vis = int(wl.cached_lens[s]) + i + 1
            dec = oracle.decode(oc.k, oc.v, q[t:t + 1], [oc.tables[s]], [n_vis], wl.scale)
            assert np.array_equal(got[t], dec[0])


def test_prefill_against_library_sdpa_causal_mask():
    wl, oc, q, cu = _prefill_case([5, 16], [9, 16], seed=72, G=2, Hkv=2, D=64)
    got = oracle.prefill(oc.k, oc.v, q, cu, wl.total_lens, oc.tables, wl.scale, causal=True)
    qf = oracle.bits_to_f64(q)
    for s in range(wl.num_seqs):
        n = int(wl.total_lens[s])
        k, v = _gathered(oc, s, n)
        c, nn = int(wl.cached_lens[s]), int(wl.new_lens[s])
        for g in range(wl.num_q_heads):
            h = g // 2
            qs = torch.from_numpy(qf[cu[s]:cu[s + 1], g])
            mask = torch.tensor([[j <= c + i for j in range(n)] for i in range(nn)])
            ref = torch.nn.functional.scaled_dot_product_attention(
                qs[None, None], torch.from_numpy(k[:, h])[None, None],
                torch.from_numpy(v[:, h])[None, None], attn_mask=mask[None, None],
                scale=wl.scale)[0, 0].numpy()
            np.testing.assert_allclose(got[cu[s]:cu[s + 1], g], ref, rtol=1e-12, atol=1e-13)


def test_prefill_non_causal_sees_everything():
    wl, oc, q, cu = _prefill_case([7], [6], seed=73, causal=False)
    got = oracle.prefill(oc.k, oc.v, q, cu, wl.total_lens, oc.tables, wl.scale, causal=False)
    for i in range(6):
        dec = oracle.decode(oc.k, oc.v, q[i:i + 1], [oc.tables[0]], [13], wl.scale)
        assert np.array_equal(got[i], dec[0])


def test_prefill_row_sampling_matches_full():
    wl, oc, q, cu = _prefill_case([10, 3], [8, 4], seed=74)
    full = oracle.prefill(oc.k, oc.v, q, cu, wl.total_lens, oc.tables, wl.scale)
    rows = [(0, 0), (7, 3), (11, 7), (9, 5)]
    part = oracle.prefill(oc.k, oc.v, q, cu, wl.total_lens, oc.tables, wl.scale, rows=rows)
    for r, (t, g) in enumerate(rows):
        assert np.array_equal(part[r], full[t, g])


# ----------------------------------------------------------------- write / copy / scenario
def test_write_lands_each_token_in_its_slot_and_leaves_the_rest():
    wl = workloads.custom_decode(3, 4, 2, 64, 4, "f32", [5, 8, 1], seed=81)
    oc = oracle.OracleCache(wl)
    written = set()
    for s in range(3):
        n = int(wl.total_lens[s])
        k, v = wl.kv_values(s, 0, n)
        for i in range(n):
            b, off = oc.tables[s][i // 4], i % 4
            assert np.array_equal(oc.k[b, :, off], k[i].numpy())
            assert np.array_equal(oc.v[b, :, off], v[i].numpy())
            written.add((b, off))
    raw = oc.k.view(np.uint32)
    for b in range(wl.num_blocks):
        for off in range(4):
            if (b, off) not in written:
                assert (raw[b, :, off] == 0xFFFFFFFF).all()


def test_write_rejects_out_of_pool_slot():
    k, v = oracle.poisoned_pool(4, 1, 2, 8, "f32")
    row = np.zeros((1, 1, 8), np.float32)
    with pytest.raises(IndexError):
        oracle.write_kv(k, v, row, row, [8])
    with pytest.raises(IndexError):
        oracle.write_kv(k, v, row, row, [-1])
    assert (k.view(np.uint32) == 0xFFFFFFFF).all()


def test_copy_blocks_copies_whole_block():
    k, v = oracle.poisoned_pool(6, 2, 4, 8, "bf16")
    src_k = np.arange(64, dtype=np.uint16).reshape(2, 4, 8)
    k[2] = src_k
    v[2] = 7
    oracle.copy_blocks(k, v, [2], [5])
    # dst holds the source's rows and the source is unchanged
    assert np.array_equal(k[5], src_k) and np.array_equal(k[2], src_k)
    assert (v[5] == 7).all() and (v[2] == 7).all()
    with pytest.raises(IndexError):
        oracle.copy_blocks(k, v, [0], [6])


def test_shared_prefix_scenario_small():
    # the long shared-prefix workload, shrunk: each pair shares its prefix
    # blocks, exactly one copy-on-write per pair, refcounts match holders
    wl = workloads.decode_long_shared(scale=1 / 512)
    oc = oracle.OracleCache(wl)
    assert len(oc.cow_pairs) == wl.num_seqs // 2
    for a in range(0, wl.num_seqs, 2):
        P = int(wl.prefix_len[a])
        full_shared = P // wl.block_size
        assert oc.tables[a][:full_shared] == oc.tables[a + 1][:full_shared]
        assert oc.tables[a][full_shared] != oc.tables[a + 1][full_shared]
    for b in range(wl.num_blocks):
        assert oc.pool.refcount[b] == _holders(oc.tables, b)
    # members agree on the shared prefix values and differ after it
    s = 0
    P = int(wl.prefix_len[s])
    ka, _ = wl.kv_values(0, 0, P + 4)
    kb, _ = wl.kv_values(1, 0, P + 4)
    assert torch.equal(ka[:P], kb[:P]) and not torch.equal(ka[P:], kb[P:])


# ----------------------------------------------------------------- sliding window
WINDOW_CASES = [
    ("f32", 2, 2, 64, 4, [1, 4, 5, 17, 40]),
    ("bf16", 4, 2, 128, 16, [1, 16, 17, 40, 70]),
    ("bf16", 8, 1, 128, 1, [33, 2, 9]),
]


@pytest.mark.parametrize("dtype,G,Hkv,D,bp,lens", WINDOW_CASES)
@pytest.mark.parametrize("window", [1, 3, 16, 17])
def test_window_decode_matches_library_sdpa_over_the_last_keys(dtype, G, Hkv, D, bp, lens, window):
    # "03｜PagedAttention 与 KV Cache 内存系统" §7: the window of position p is [p - w + 1, p]
    wl, oc, q = _small_case(dtype, G, Hkv, D, bp, lens, seed=window + len(lens))
    got = oracle.decode_window(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale, window)
    qf = oracle.bits_to_f64(q)
    for s, n in enumerate(wl.total_lens):
        k, v = _gathered(oc, s, int(n))
        lo = max(0, int(n) - window)
        for g in range(wl.num_q_heads):
            h = g // G
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(qf[s, g][None, None, None]),
                torch.from_numpy(k[lo:, h][None, None]),
                torch.from_numpy(v[lo:, h][None, None]), scale=wl.scale)[0, 0, 0].numpy()
            np.testing.assert_allclose(got[s, g], ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("window", [0, -1, 70, 1000])
def test_window_wider_than_the_context_is_full_decode_bit_for_bit(window):
    wl, oc, q = _small_case("bf16", 4, 2, 128, 16, [1, 16, 17, 40, 70], seed=5)
    full = oracle.decode(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale)
    got = oracle.decode_window(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale, window)
    assert np.array_equal(got, full)


def test_window_of_one_returns_the_newest_value_exactly():
    wl, oc, q = _small_case("f32", 2, 2, 64, 4, [1, 5, 17], seed=8)
    got = oracle.decode_window(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale, 1)
    for s, n in enumerate(wl.total_lens):
        _, v = _gathered(oc, s, int(n))
        for g in range(wl.num_q_heads):
            assert np.array_equal(got[s, g], v[int(n) - 1, g // 2])


def test_window_rows_match_full_window_result():
    wl, oc, q = _small_case("bf16", 4, 2, 128, 16, [40, 70], seed=6)
    full = oracle.decode_window(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale, 20)
    rows = [(1, 7), (0, 0), (1, 3)]
    got = oracle.decode_window(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale, 20, rows=rows)
    for r, (s, g) in enumerate(rows):
        assert np.array_equal(got[r], full[s, g])

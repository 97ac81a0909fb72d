"""GPU parity of pa_decode_shared (shared-prefix-aware decode) against the float64 oracle.

Reading a pair's shared pages once changes where the bytes come from, not
the result, so the oracle is the plain decode definition (oracle.decode) over
the same tables.  Tolerance as for every bf16 decode: max |err| <= 2e-3 and
relative L2 <= 1e-3 on the fp32 outputs.  Inconsistent pair declarations
are flagged with PA_ERR_INVALID_ARG and decoded on their own (still within
tolerance).
"""
import dataclasses

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


def _declared(wl):
    """partner / shared_lens of the workload's pairs: the whole shared pages
    of each prefix (the partial tail page was copied on write)."""
    B = wl.num_seqs
    partner = np.full(B, -1, np.int32)
    shared = np.zeros(B, np.int32)
    if wl.pair_of is not None:
        for s in range(B):
            q = int(wl.pair_of[s])
            if q >= 0:
                partner[s] = q
                shared[s] = int(wl.prefix_len[s]) // wl.block_size * wl.block_size
    return partner, shared


def _decode_shared(g, partner, shared, part=0):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(g.device)
    g.err.zero_()
    out = pkv.decode_shared(g.cache.pool, g.q, g.block_tables, g.context_lens, g.max_context,
                            t(partner), t(shared), g.wl.scale, partition_tokens=part,
                            d_err=g.err)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(g.err.item())


def _setup(wl):
    g = GpuWorkload(wl)
    g.write_new()
    tables = g.tables_list()
    partner, shared = _declared(wl)
    for s in range(wl.num_seqs):  # the declared pages really are shared
        if partner[s] >= 0:
            k = int(shared[s]) // wl.block_size
            assert tables[s][:k] == tables[partner[s]][:k]
    oc = oracle.OracleCache(wl)
    ref = oracle.decode(oc.k, oc.v, oracle.to_numpy_bits(g.q_host), oc.tables, wl.total_lens,
                        wl.scale)
    return g, partner, shared, ref


def _long_shared(scale, G=8, block_size=16, pairs="adjacent"):
    wl = workloads.decode_long_shared(scale, pairs=pairs)
    return dataclasses.replace(wl, num_q_heads=G * wl.num_kv_heads, block_size=block_size)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("part", [0, 32, 48])
def test_shared_decode_matches_oracle(G, part):
    g, partner, shared, ref = _setup(_long_shared(1 / 64, G))
    got, err = _decode_shared(g, partner, shared, part)
    assert err == 0, pkv.status_str(err)
    _check(got, ref, "G=%d part=%d" % (G, part))


@pytest.mark.parametrize("block_size", [32, 64])
@pytest.mark.parametrize("pairs", ["adjacent", "far"])
def test_shared_decode_block_sizes_and_pair_placement(block_size, pairs):
    g, partner, shared, ref = _setup(_long_shared(1 / 64, 8, block_size, pairs))
    got, err = _decode_shared(g, partner, shared)
    assert err == 0, pkv.status_str(err)
    _check(got, ref, "bp=%d %s" % (block_size, pairs))


def test_shared_decode_without_pairs_is_plain_decode():
    g, partner, shared, ref = _setup(_long_shared(1 / 64))
    got, err = _decode_shared(g, np.full_like(partner, -1), np.zeros_like(shared))
    assert err == 0
    _check(got, ref, "no pairs declared")
    # a batch without any sharing at all
    g2, p2, s2, ref2 = _setup(workloads.decode_gqa(scale=1 / 8))
    got2, err2 = _decode_shared(g2, p2, s2)
    assert err2 == 0
    _check(got2, ref2, "decode_gqa, no pairs")


def _bad_declarations(partner, shared, block_size):
    a, b = 0, int(partner[0])
    cases = []
    p = partner.copy()
    p[b] = -1  # not mutual
    cases.append(("one-sided", p, shared.copy()))
    s = shared.copy()
    s[b] -= block_size  # the two sides disagree on the length
    cases.append(("length mismatch", partner.copy(), s))
    s = shared.copy()
    s[a] = s[b] = shared[a] - 8  # not a multiple of the block size
    cases.append(("unaligned length", partner.copy(), s))
    s = shared.copy()
    s[a] = s[b] = 1 << 30  # longer than the contexts
    cases.append(("too long", partner.copy(), s))
    p = partner.copy()
    p[a] = p[b] = a  # a sequence paired with itself
    cases.append(("self pair", p, shared.copy()))
    p = partner.copy()
    p[a] = 1 << 20  # outside the batch
    cases.append(("partner outside batch", p, shared.copy()))
    return cases


def test_shared_decode_flags_inconsistent_declarations_and_stays_correct():
    wl = _long_shared(1 / 64)
    g, partner, shared, ref = _setup(wl)
    for what, p, s in _bad_declarations(partner, shared, wl.block_size):
        got, err = _decode_shared(g, p, s)
        assert err == pkv.PA_ERR_INVALID_ARG, what
        _check(got, ref, what)


def test_shared_decode_flags_tables_that_differ_over_declared_pages():
    # declare the pages of two unrelated sequences as shared
    wl = workloads.decode_gqa(scale=1 / 8)
    g = GpuWorkload(wl)
    g.write_new()
    partner = np.full(wl.num_seqs, -1, np.int32)
    shared = np.zeros(wl.num_seqs, np.int32)
    partner[0], partner[1] = 1, 0
    shared[0] = shared[1] = 64
    _, err = _decode_shared(g, partner, shared)
    assert err == pkv.PA_ERR_INVALID_ARG


def test_shared_decode_rejects_unsupported_pools():
    # pages of 8 tokens: a 16-token chunk would span two pages
    wl = workloads.custom_decode(4, 8, 2, 128, 8, "bf16", [40, 40, 40, 40], seed=3)
    g = GpuWorkload(wl)
    partner = np.array([1, 0, -1, -1], np.int32)
    shared = np.array([16, 16, 0, 0], np.int32)
    with pytest.raises(pkv.PagedKVError) as e:
        _decode_shared(g, partner, shared)
    assert e.value.status == pkv.PA_ERR_UNSUPPORTED


@pytest.mark.parametrize("pairs", ["adjacent", "far"])
def test_shared_decode_full_size_sampled(pairs):
    wl = workloads.decode_long_shared(pairs=pairs)
    g = GpuWorkload(wl)
    g.write_new()
    partner, shared = _declared(wl)
    got, err = _decode_shared(g, partner, shared)
    assert err == 0, pkv.status_str(err)
    plain = pkv.decode(g.cache.pool, g.q, g.block_tables, g.context_lens, g.max_context,
                       wl.scale).cpu().numpy()
    oc = oracle.OracleCache(wl)
    rng = np.random.default_rng(11)
    rows = [(int(s), int(h)) for s, h in zip(rng.integers(0, wl.num_seqs, 64),
                                             rng.integers(0, wl.num_q_heads, 64))]
    rows += [(s, 0) for s in range(wl.num_seqs)]
    ref = oracle.decode(oc.k, oc.v, oracle.to_numpy_bits(g.q_host), oc.tables, wl.total_lens,
                        wl.scale, rows=rows)
    _check(np.stack([got[s, h] for s, h in rows]), ref, "full size %s" % pairs)
    _check(got, plain, "against pa_decode")

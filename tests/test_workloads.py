"""The seeded synthetic inputs follow the recipe that workloads.py states in
its module docstring: shapes, length distributions, pool sizing, the
shared-prefix construction, and reproducible N(0, 1) values."""
import math

import numpy as np
import torch

import workloads


def _blocks(n, bp):
    return int((-(-np.asarray(n, np.int64) // bp)).sum())


def test_shapes_and_scales():
    want = {  # B, H_q, H_kv, D, B_p, dtype
        "decode_tiny": (4, 4, 2, 64, 4, "f32"),
        "decode_gqa": (64, 32, 8, 128, 16, "bf16"),
        "decode_mha": (256, 32, 32, 128, 16, "bf16"),
        "decode_long_shared": (8, 64, 8, 128, 16, "bf16"),
        "prefill": (16, 32, 8, 128, 16, "bf16"),
    }
    for name, shape in want.items():
        wl = workloads.WORKLOADS[name]()
        got = (wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size, wl.dtype)
        assert got == shape, name
        assert wl.scale == 1.0 / math.sqrt(wl.head_dim)
        assert np.array_equal(np.sort(wl.free_order), np.arange(wl.num_blocks)), name


def test_length_distributions():
    tiny = workloads.decode_tiny()
    assert tiny.cached_lens.min() >= 1 and tiny.cached_lens.max() <= 64
    gqa = workloads.decode_gqa()
    assert gqa.cached_lens.min() >= 128 and gqa.cached_lens.max() <= 4096
    assert 1500 < gqa.cached_lens.mean() < 2700           # U[128, 4096]: mean 2112
    mha = workloads.decode_mha()
    c = mha.cached_lens
    assert c.min() >= 16 and c.max() <= 2048
    assert 350 < np.median(c) < 750                        # lognormal(ln 512, 1): median 512
    ls = workloads.decode_long_shared()
    assert ls.cached_lens.min() >= 32768 and ls.cached_lens.max() <= 131072
    pf = workloads.prefill()
    assert np.all(pf.cached_lens == 2048) and np.all(pf.new_lens == 512) and pf.causal
    for wl in (tiny, gqa, mha, ls):
        assert np.all(wl.new_lens == 1) and wl.kind == "decode"


def test_pool_sizing():
    for make in (workloads.decode_gqa, workloads.decode_mha, workloads.prefill):
        wl = make()
        need = _blocks(wl.total_lens, wl.block_size)
        assert wl.num_blocks == int(math.floor(1.5 * need)), wl.name
    assert workloads.decode_tiny().num_blocks == 128
    ls = workloads.decode_long_shared()
    need = _blocks(ls.total_lens, 16)
    assert ls.num_blocks == max(int(math.floor(1.1 * need)), need + 64)


def test_shared_prefix_construction():
    wl = workloads.decode_long_shared()
    assert list(wl.pair_of) == [1, 0, 3, 2, 5, 4, 7, 6]
    for a in range(0, 8, 2):
        b = a + 1
        p = int(wl.prefix_len[a])
        assert p == int(wl.prefix_len[b])
        full = int(math.floor(0.75 * min(wl.cached_lens[a], wl.cached_lens[b])))
        assert p in (full, full - 1) and p % 16 != 0      # the shared tail block is partial
        assert p < min(wl.cached_lens[a], wl.cached_lens[b])


def test_values_are_reproducible_and_shared_below_the_prefix():
    wl = workloads.decode_long_shared(scale=1 / 256)
    wl2 = workloads.decode_long_shared(scale=1 / 256)
    assert np.array_equal(wl.cached_lens, wl2.cached_lens)
    assert np.array_equal(wl.free_order, wl2.free_order)
    a, b = 0, 1
    p = int(wl.prefix_len[a])
    ka, va = wl.kv_values(a, 0, int(wl.cached_lens[a]))
    kb, vb = wl2.kv_values(b, 0, int(wl2.cached_lens[b]))
    assert torch.equal(ka[:p], kb[:p]) and torch.equal(va[:p], vb[:p])
    assert not torch.equal(ka[p:p + 8], kb[p:p + 8])
    # any window is the same slice of the whole sequence
    assert torch.equal(wl.kv_values(a, 5, 70)[0], ka[5:70])
    assert torch.equal(wl.queries(), wl2.queries())


def test_values_are_standard_normal_rounded_to_the_storage_dtype():
    wl = workloads.decode_gqa(scale=1 / 8)
    k, v = wl.kv_values(0, 0, int(wl.cached_lens[0]))
    assert k.dtype == torch.bfloat16 and v.dtype == torch.bfloat16
    x = torch.cat([k.flatten(), v.flatten()]).double()
    assert abs(float(x.mean())) < 0.02 and abs(float(x.std()) - 1.0) < 0.02
    q = workloads.decode_tiny().queries()
    assert q.dtype == torch.float32 and tuple(q.shape) == (4, 4, 64)

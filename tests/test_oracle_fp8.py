"""Pins of the oracle's FP8 (E4M3) page format (oracle/fp8.py) against the OCP
8-bit floating point definition, a library conversion and closed-form error
bounds, and of the float64-pool attention path it uses."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import fp8


def test_decode_table_values_from_the_definition():
    # S.EEEE.MMM, bias 7: code 0x38 = 1.0, 0x08 = 2^-6 (smallest normal),
    # 0x01 = 2^-9 (smallest subnormal), 0x7E = 1.75 * 2^8 = 448, 0x7F = NaN
    v = fp8.e4m3_decode([0x00, 0x01, 0x07, 0x08, 0x38, 0x39, 0x7E, 0x7F, 0x80, 0xB8, 0xFE, 0xFF])
    assert v[0] == 0.0 and v[1] == 2.0 ** -9 and v[2] == 7 * 2.0 ** -9
    assert v[3] == 2.0 ** -6 and v[4] == 1.0 and v[5] == 1.125 and v[6] == 448.0
    assert np.isnan(v[7]) and np.isnan(v[11])
    assert v[8] == 0.0 and np.signbit(v[8]) and v[9] == -1.0 and v[10] == -448.0
    allv = fp8.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert np.isnan(allv).sum() == 2
    assert np.all(np.diff(allv[:0x7F]) > 0)           # positive codes increase
    assert np.array_equal(allv[0x80:0xFF], -allv[:0x7F])  # sign-magnitude


def test_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(fp8.e4m3_encode(fp8.e4m3_decode(codes)), codes)


def test_encode_rounds_to_nearest_even_and_saturates():
    x = [1.0625, 1.1875, 1.0624, 1.0626, 2.0 ** -10, 3 * 2.0 ** -10, 464.0, 1e9, -1e9,
         float("inf"), -float("inf"), float("nan")]
    got = fp8.e4m3_encode(x)
    # ties go to the even mantissa, 464 (the would-be next step) saturates to 448
    assert list(got) == [0x38, 0x3A, 0x38, 0x39, 0x00, 0x02, 0x7E, 0x7E, 0xFE, 0x7E, 0xFE, 0x7F]


def test_encode_matches_the_library_conversion_in_range():
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch has no float8_e4m3fn")
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.uniform(-448, 448, 20000), rng.normal(0, 1, 20000),
                        rng.normal(0, 0.01, 20000)]).astype(np.float32)
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.e4m3_encode(x), lib)


def test_row_quantisation_error_bound_and_scale():
    rng = np.random.default_rng(5)
    x = rng.normal(0, 1, (64, 8, 128)).astype(np.float32)
    x[0, 0] = 0.0                                  # an all-zero row
    codes, scales = fp8.quantize_rows(x)
    amax = np.abs(x).max(-1)
    assert np.array_equal(scales, (amax / np.float32(448)).astype(np.float32))
    deq = fp8.dequantize(codes, scales)
    assert np.all(deq[0, 0] == 0.0)
    # in code units y = x * 448 / amax the rounding error is at most half a step:
    # 2^-4 |y| for normals, 2^-10 below 2^-6; plus the rounding of 448/amax
    y = np.abs(x.astype(np.float64)) * 448.0 / np.maximum(amax, 1e-30)[..., None]
    bound = np.maximum(2.0 ** -4 * y, 2.0 ** -10) * scales[..., None] + 1e-6 * np.abs(x)
    assert np.all(np.abs(deq - x) <= bound + 1e-30)
    # the largest element of every non-zero row lands on +-448 (or next to it)
    top = np.abs(fp8.e4m3_decode(codes)).max(-1)
    assert np.all((top[amax > 0] >= 416.0) & (top[amax > 0] <= 448.0))


def test_float64_pool_attention_equals_bf16_pool_attention():
    wl = workloads.custom_decode(5, 8, 2, 128, 16, "bf16", [0, 15, 16, 40, 99], seed=12)
    oc = oracle.OracleCache(wl)
    q = oracle.to_numpy_bits(wl.queries())
    ref = oracle.decode(oc.k, oc.v, q, oc.tables, wl.total_lens, wl.scale)
    got = oracle.decode(oracle.bits_to_f64(oc.k), oracle.bits_to_f64(oc.v),
                        oracle.bits_to_f64(q), oc.tables, wl.total_lens, wl.scale)
    assert np.array_equal(got, ref)


def test_write_then_slot_quantisation_agree():
    # write_kv_fp8 row by row gives the same pools as quantising the bf16 pool
    wl = workloads.custom_decode(3, 8, 2, 128, 16, "bf16", [5, 20, 33], seed=4)
    oc = oracle.OracleCache(wl)
    kc, vc, ks, vs = fp8.fp8_pools_from(oc.k, oc.v)
    kc2, vc2, ks2, vs2 = fp8.poisoned_fp8_pool(wl.num_blocks, wl.num_kv_heads, wl.block_size,
                                              wl.head_dim)
    for s, table in enumerate(oc.tables):
        n = int(wl.total_lens[s])
        slots = [table[i // wl.block_size] * wl.block_size + i % wl.block_size for i in range(n)]
        rows_k = np.stack([oracle.bits_to_f64(oc.k[sl // 16, :, sl % 16]) for sl in slots])
        rows_v = np.stack([oracle.bits_to_f64(oc.v[sl // 16, :, sl % 16]) for sl in slots])
        fp8.write_kv_fp8(kc2, vc2, ks2, vs2, rows_k.astype(np.float32),
                         rows_v.astype(np.float32), slots)
    assert np.array_equal(kc, kc2) and np.array_equal(vc, vc2)
    assert np.array_equal(ks, ks2, equal_nan=True) and np.array_equal(vs, vs2, equal_nan=True)

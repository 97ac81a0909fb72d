"""FP8 (E4M3) KV pages for the oracle: encoding, per-row scales, dequantisation.

TEST INFRASTRUCTURE, like the rest of ``oracle/``.

The pages say that quantised KV pages carry their scales inside the page
budget ("KV Cache：容量、布局与生命周期", the capacity formula with the dtype's
bytes per element; "03｜PagedAttention 与 KV Cache 内存系统" §1.1 and §6 on
quantisation as an optimisation on top of paging) but fix no format.  The
reading taken here: E4M3 codes as defined by the OCP 8-bit floating point
specification (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
exponent field 0 is subnormal; S.1111.111 is NaN; no infinities; largest
finite magnitude 448), one float32 scale per (token, kv-head) row:

    amax  = max_d |x_d|                       (float32)
    scale = amax / 448                        (float32 division, rounded)
    inv   = 448 / amax                        (float32 division, rounded; 0 if amax == 0)
    code_d = E4M3(x_d * inv)                  (float32 product, then round to
                                               nearest, ties to even, saturating
                                               to +-448)
    value_d = decode(code_d) * scale          (exact in float64)

Attention over an FP8 pool is then the ordinary attention of ``attention.c``
over the dequantised values, in float64.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
NAN_CODE = 0x7F


def e4m3_decode(codes) -> np.ndarray:
    """uint8 E4M3 codes -> float64 values (NaN for S.1111.111)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    out = sign * mag
    return np.where((e == 15) & (m == 7), np.nan, out)


# the 127 non-negative finite magnitudes, in code order (codes 0x00 .. 0x7E),
# which is also increasing order
_POS_CODES = np.arange(0x7F, dtype=np.uint8)
_POS_VALUES = e4m3_decode(_POS_CODES)
assert np.all(np.diff(_POS_VALUES) > 0)


def e4m3_encode(x) -> np.ndarray:
    """float values -> uint8 E4M3 codes: nearest representable magnitude, ties to
    the even code (mantissa LSB 0), magnitudes above 448 (and infinities)
    saturate to 448, NaN -> 0x7F; the sign bit is kept (-0.0 -> 0x80)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    a_sat = np.minimum(np.where(np.isnan(a), 0.0, a), E4M3_MAX)
    hi = np.searchsorted(_POS_VALUES, a_sat, side="left")  # first value >= a
    hi = np.minimum(hi, len(_POS_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    v_lo, v_hi = _POS_VALUES[lo], _POS_VALUES[hi]
    d_lo, d_hi = a_sat - v_lo, v_hi - a_sat
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((hi & 1) == 0))
    code = np.where(a_sat >= v_hi, hi, np.where(pick_hi, hi, lo)).astype(np.uint8)
    code = code | np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(NAN_CODE), code).astype(np.uint8)


def quantize_rows(x):
    """Rows [..., D] of float32 values -> (codes uint8 [..., D], scales float32 [...])."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1)
    with np.errstate(divide="ignore"):
        scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
        inv = np.where(amax > 0, np.float32(E4M3_MAX) / amax, np.float32(0)).astype(np.float32)
    y = (x * inv[..., None]).astype(np.float32)
    return e4m3_encode(y), scale


def dequantize(codes, scales) -> np.ndarray:
    """codes [..., D] and scales [...] -> float64 values."""
    return e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[..., None]


def poisoned_fp8_pool(num_blocks: int, num_kv_heads: int, block_size: int, head_dim: int):
    """K and V code pools [N][H][B_p][D] and their scale pools [N][H][B_p] with every
    byte 0xFF (code 0xFF is a NaN, and so are the scales): the same poison as the
    bf16/f32 pools, so a read of an unwritten slot shows up."""
    shape = (num_blocks, num_kv_heads, block_size, head_dim)
    kc = np.full(shape, 0xFF, dtype=np.uint8)
    vc = np.full(shape, 0xFF, dtype=np.uint8)
    ks = np.full(shape[:3], 0xFFFFFFFF, dtype=np.uint32).view(np.float32)
    vs = np.full(shape[:3], 0xFFFFFFFF, dtype=np.uint32).view(np.float32)
    return kc, vc, ks, vs


def write_kv_fp8(kcodes, vcodes, kscales, vscales, k_new, v_new, slot_mapping):
    """Quantise and scatter one K and one V row per (token, kv-head) into its slot
    (the write path of P1 §4.1 with FP8 pages).  k_new/v_new: float32 [T][H][D]."""
    N, H, Bp, D = kcodes.shape
    kq, ksc = quantize_rows(k_new)
    vq, vsc = quantize_rows(v_new)
    for t, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot < 0 or slot >= N * Bp:
            raise IndexError("slot %d outside the pool" % slot)
        blk, off = divmod(slot, Bp)
        kcodes[blk, :, off, :] = kq[t]
        vcodes[blk, :, off, :] = vq[t]
        kscales[blk, :, off] = ksc[t]
        vscales[blk, :, off] = vsc[t]


def fp8_pools_from(kpool, vpool):
    """The FP8 pools that writing the same rows through write_kv_fp8 produces,
    from an oracle pool of float32 or bf16 bits (every slot holds the last row
    written to it, so quantising slot by slot is the same as quantising at
    write time); slots never written (NaN-poisoned rows) keep the poison of
    poisoned_fp8_pool."""
    from . import bits_to_f64
    N, H, Bp, D = kpool.shape
    kc, vc, ks, vs = poisoned_fp8_pool(N, H, Bp, D)
    for src, codes, scales in ((kpool, kc, ks), (vpool, vc, vs)):
        f = bits_to_f64(src).astype(np.float32)
        written = ~np.isnan(f).any(axis=-1)
        q, sc = quantize_rows(np.where(written[..., None], f, np.float32(0)))
        codes[written] = q[written]
        scales[written] = sc[written]
    return kc, vc, ks, vs


def dequantized_pools(kcodes, vcodes, kscales, vscales):
    """float64 K and V pools holding decode(code) * scale (for attention.c, dtype 2)."""
    return dequantize(kcodes, kscales), dequantize(vcodes, vscales)

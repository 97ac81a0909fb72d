"""Host-side argument checks of the Python binding: shapes, dtypes and the
device error word are rejected before anything reaches the C ABI (a
wrong-shaped output or a host error word would otherwise become an
out-of-bounds device write).  Runs on the CPU: the checks raise before any
library call."""
import pytest
import torch

import paged_kv_cache_148_gb300 as pkv


def _pool():
    return pkv.KVPool(8, 16, 2, 128, torch.bfloat16, device="cpu")


def _decode_args(B=3, Hq=8, D=128, max_blocks=4):
    return dict(q=torch.zeros(B, Hq, D, dtype=torch.bfloat16),
                block_tables=torch.zeros(B, max_blocks, dtype=torch.int32),
                context_lens=torch.ones(B, dtype=torch.int32))


def _decode(pool, **kw):
    a = _decode_args()
    a.update(kw)
    return pkv.decode(pool, a["q"], a["block_tables"], a["context_lens"], 64, 0.1,
                      out=a.get("out"), d_err=a.get("d_err"), phase=a.get("phase", "all"))


@pytest.mark.parametrize("bad,exc", [
    (dict(out=torch.zeros(3, 8, 64)), ValueError),                  # wrong out shape
    (dict(out=torch.zeros(3, 8, 128, dtype=torch.float64)), TypeError),
    (dict(q=torch.zeros(3, 8, 64, dtype=torch.bfloat16)), ValueError),   # D != head_dim
    (dict(q=torch.zeros(3, 8, 128, dtype=torch.float32)), TypeError),    # not the pool dtype
    (dict(context_lens=torch.ones(2, dtype=torch.int32)), ValueError),
    (dict(block_tables=torch.zeros(2, 4, dtype=torch.int32)), ValueError),
    (dict(block_tables=torch.zeros(3, 4, dtype=torch.int64)), TypeError),
    (dict(d_err=torch.zeros(1, dtype=torch.int64)), TypeError),
    (dict(d_err=torch.zeros(0, dtype=torch.int32)), ValueError),
    (dict(phase="both"), ValueError),
])
def test_decode_rejects_bad_arguments(bad, exc):
    with pytest.raises(exc):
        _decode(_pool(), **bad)


def test_window_and_step_share_the_decode_checks():
    pool, a = _pool(), _decode_args()
    with pytest.raises(ValueError):
        pkv.decode_window(pool, a["q"], a["block_tables"], a["context_lens"], 64, 16, 0.1,
                          out=torch.zeros(3, 8, 127))
    k_new = torch.zeros(3, 2, 128, dtype=torch.bfloat16)
    slots = torch.zeros(3, dtype=torch.int64)
    with pytest.raises(ValueError):
        pkv.decode_step(pool, k_new, k_new, slots, a["q"], a["block_tables"],
                        torch.ones(4, dtype=torch.int32), 64, 0.1, None)
    with pytest.raises(TypeError):
        pkv.decode_step(pool, k_new, k_new, slots, a["q"], a["block_tables"], a["context_lens"],
                        64, 0.1, None, d_err=torch.zeros(1, dtype=torch.float32))


def test_prefill_rejects_bad_shapes():
    pool = _pool()
    T, B = 10, 2
    q = torch.zeros(T, 8, 128, dtype=torch.bfloat16)
    cu = torch.tensor([0, 4, 10], dtype=torch.int32)
    lens = torch.tensor([20, 30], dtype=torch.int32)
    bt = torch.zeros(B, 4, dtype=torch.int32)
    with pytest.raises(ValueError):   # cu_seqlens_q must be [B + 1]
        pkv.prefill(pool, q, cu[:2], lens, bt, 6, 30, 0.1)
    with pytest.raises(ValueError):   # block_tables rows != B
        pkv.prefill(pool, q, cu, lens, bt[:1], 6, 30, 0.1)
    with pytest.raises(ValueError):   # out must be [T][H_q][D]
        pkv.prefill(pool, q, cu, lens, bt, 6, 30, 0.1, out=torch.zeros(T - 1, 8, 128))
    with pytest.raises(TypeError):
        pkv.prefill(pool, q, cu, lens, bt, 6, 30, 0.1, d_err=torch.zeros(1, dtype=torch.int16))


def test_write_and_copy_check_the_error_word():
    pool = _pool()
    k = torch.zeros(4, 2, 128, dtype=torch.bfloat16)
    slots = torch.zeros(4, dtype=torch.int64)
    with pytest.raises(TypeError):
        pkv.write_kv(pool, k, k, slots, d_err=torch.zeros(1, dtype=torch.int64))
    ids = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(ValueError):
        pkv.copy_blocks(pool, ids, ids, d_err=torch.zeros(0, dtype=torch.int32))

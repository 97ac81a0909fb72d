"""pa_decode_noalloc: decode with no caller-provided workspace.

Callers that cannot allocate device memory when they run decode (code being
captured into a CUDA graph, plugin hosts that hand over raw pointers but no
allocator, processes whose HBM all belongs to the block pool) use this entry
point; its split-KV scratch lives in a static device array inside the
library.  The test calls it through the C ABI twice in a row and checks each
result against pa_decode with an ordinary workspace, within the same bf16
tolerance as the other decode tests.  It runs on its own in a fresh process
as well as after the other tests, and is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

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


def _noalloc(g, out, partition_tokens, err):
    wl = g.wl
    return pkv.lib().pa_decode_noalloc(
        g.cache.pool.c, ctypes.c_void_p(g.q.data_ptr()), wl.num_q_heads,
        ctypes.c_void_p(g.block_tables.data_ptr()), int(g.block_tables.shape[1]),
        ctypes.c_void_p(g.context_lens.data_ptr()), wl.num_seqs, g.max_context,
        ctypes.c_float(wl.scale), partition_tokens, ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(err.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_decode_matches_workspace_decode_on_two_calls():
    wl = workloads.decode_gqa(scale=1 / 4)
    g = GpuWorkload(wl)
    g.write_new()
    part = 64  # several partitions per sequence, so the static scratch is used
    assert pkv.decode_workspace_bytes(g.cache.pool, wl.num_seqs, wl.num_q_heads,
                                      g.max_context, part) > 0
    g.set_partition_tokens(part)
    ref = g.attend().clone()
    torch.cuda.synchronize()
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        st = _noalloc(g, out, part, err)
        assert st == pkv.PA_OK, pkv.status_str(st)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        a, b = out.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64)
        assert np.isfinite(a).all()
        assert np.abs(a - b).max() <= MAX_ABS
        assert np.linalg.norm(a - b) / np.linalg.norm(b) <= REL_L2


def test_noalloc_rejects_shapes_beyond_the_static_scratch():
    wl = workloads.decode_gqa(scale=1 / 16)
    g = GpuWorkload(wl)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(g.out)
    # 16-token partitions over a 2^20-token context need far more than 16 MiB
    st = pkv.lib().pa_decode_noalloc(
        g.cache.pool.c, ctypes.c_void_p(g.q.data_ptr()), wl.num_q_heads,
        ctypes.c_void_p(g.block_tables.data_ptr()), int(g.block_tables.shape[1]),
        ctypes.c_void_p(g.context_lens.data_ptr()), wl.num_seqs, 1 << 20,
        ctypes.c_float(wl.scale), 16, ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(err.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == pkv.PA_ERR_UNSUPPORTED

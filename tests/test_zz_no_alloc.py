"""pa_decode_noalloc: decode with no caller-provided workspace.

Some callers cannot allocate device memory when they run decode: plugin or
custom-op hosts that hand over raw device pointers but no allocator, and
serving processes that give all spare HBM to the block pool.  They use this
entry point; its split-KV scratch lives in a static device array inside the
library.  The tests call it through the C ABI twice in a row.  Both calls
must equal pa_decode with an ordinary workspace bit for bit, since they run
the same kernels with the same partition plan.  Both must also match the
float64 oracle within the bf16 decode tolerance.  One test repeats the check
in a fresh Python process, so it also covers the first call's set-up.  The
file is collected last.
"""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_148_gb300 as pkv
import workloads
from harness import GpuWorkload

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 2e-3, 1e-3
_CHILD = "PKV_NOALLOC_FRESH_PROCESS"


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
    g.err.zero_()
    ref = g.attend().clone()
    torch.cuda.synchronize()
    assert int(g.err.item()) == 0
    oc = oracle.OracleCache(wl)
    exact = oracle.decode(oc.k, oc.v, oracle.to_numpy_bits(g.q_host), oc.tables, wl.total_lens,
                          wl.scale)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        st = _noalloc(g, out, part, err)
        assert st == pkv.PA_OK, pkv.status_str(st)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, pkv.status_str(int(err.item()))
        assert torch.equal(out, ref), "call %d differs from pa_decode" % call
        a = out.cpu().numpy().astype(np.float64)
        assert np.isfinite(a).all()
        assert np.abs(a - exact).max() <= MAX_ABS
        assert np.linalg.norm(a - exact) / np.linalg.norm(exact) <= REL_L2


@pytest.mark.skipif(os.environ.get(_CHILD) == "1", reason="already the fresh process")
def test_noalloc_in_a_fresh_process():
    """The two-call check again, as the first use of the library in a new process."""
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, **{_CHILD: "1"})
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.abspath(__file__) +
                        "::test_noalloc_decode_matches_workspace_decode_on_two_calls"],
                       cwd=os.path.dirname(here), env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "1 passed" in r.stdout


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

"""Paged KV-cache attention for GB300 (sm_103a): Python binding of libpagedkv.so.

The binding only marshals arguments: it checks tensor dtype, device and
contiguity and passes raw pointers, sizes and the current CUDA stream to the
C ABI declared in ``include/pagedkv.h``.  Every step of the path runs in the
library's kernels; if the library is missing this module raises instead of
computing anything another way.

Entry points (same names as the C ABI, without the ``pa_`` prefix):
``write_kv``, ``copy_blocks``, ``decode``, ``prefill``, ``physical_slot``,
``slot_mapping``, ``page_size_bytes``, ``decode_partition_tokens``,
``decode_workspace_bytes`` and the host block ``Allocator``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedkv.so")

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_OUT_OF_RANGE = 2
PA_ERR_NEGATIVE_BLOCK = 3
PA_ERR_NO_FREE_BLOCK = 4
PA_ERR_REFCOUNT = 5
PA_ERR_UNSUPPORTED = 6
PA_ERR_CUDA = 7
PA_ERR_TIMEOUT = 8

DTYPE_F32 = 0
DTYPE_BF16 = 1
DTYPE_FP8_E4M3 = 2

EXPORTED = [
    "pa_status_str", "pa_last_cuda_error", "pa_abi_version", "pa_page_size_bytes",
    "pa_physical_slot", "pa_slot_mapping", "pa_write_kv", "pa_copy_blocks",
    "pa_decode_partition_tokens", "pa_decode_workspace_bytes", "pa_decode", "pa_decode_partial",
    "pa_decode_merge", "pa_decode_noalloc", "pa_decode_step_workspace_bytes", "pa_decode_step",
    "pa_decode_window_workspace_bytes", "pa_decode_window", "pa_decode_shared_workspace_bytes",
    "pa_decode_shared",
    "pa_prefill",
    "pa_alloc_create", "pa_alloc_destroy", "pa_alloc_append", "pa_alloc_fork",
    "pa_alloc_writable_tail", "pa_alloc_reserve", "pa_alloc_release", "pa_alloc_refcount",
    "pa_alloc_num_free",
]


class PagedKVError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


class pa_kv_pool(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("k_scale", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p)]


_lib = None


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libpagedkv.so in-tree (nvcc, sm_103a)."""
    from . import builder
    return builder.build(force=force, verbose=verbose)


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libpagedkv.so is not built (run paged_kv_cache_148_gb300.build()); "
                           "there is no fallback path")
    L = ctypes.CDLL(LIB_PATH)
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    sz = ctypes.c_size_t
    sig = {
        "pa_status_str": ([i32], ctypes.c_char_p),
        "pa_last_cuda_error": ([], ctypes.c_char_p),
        "pa_abi_version": ([], i32),
        "pa_page_size_bytes": ([P, P], i32),
        "pa_physical_slot": ([P, i32, i32, i64, P], i32),
        "pa_slot_mapping": ([P, i32, i32, P, i64, P], i32),
        "pa_write_kv": ([P, P, P, P, i32, P, P], i32),
        "pa_copy_blocks": ([P, P, P, i32, P, P], i32),
        "pa_decode_partition_tokens": ([P, i32, i32, i32, P], i32),
        "pa_decode_workspace_bytes": ([P, i32, i32, i32, i32, P], i32),
        "pa_decode": ([P, P, i32, P, i32, P, i32, i32, f32, i32, P, P, sz, P, P], i32),
        "pa_decode_partial": ([P, P, i32, P, i32, P, i32, i32, f32, i32, P, P, sz, P, P], i32),
        "pa_decode_merge": ([P, i32, P, i32, i32, i32, P, P, sz, P], i32),
        "pa_decode_noalloc": ([P, P, i32, P, i32, P, i32, i32, f32, i32, P, P, P], i32),
        "pa_decode_step_workspace_bytes": ([P, i32, i32, i32, i32, P], i32),
        "pa_decode_window_workspace_bytes": ([P, i32, i32, i32, i32, i32, P], i32),
        "pa_decode_window": ([P, P, i32, P, i32, P, i32, i32, i32, f32, i32, P, P, sz, P, P], i32),
        "pa_decode_step": ([P, P, P, P, P, i32, P, i32, P, i32, i32, f32, i32, P, P, sz, P, P], i32),
        "pa_decode_shared_workspace_bytes": ([P, i32, i32, i32, i32, P], i32),
        "pa_decode_shared": ([P, P, i32, P, i32, P, i32, i32, P, P, f32, i32, P, P, sz, P, P], i32),
        "pa_prefill": ([P, P, i32, i32, P, P, P, i32, i32, i32, i32, f32, i32, P, P, P], i32),
        "pa_alloc_create": ([i32, P, P], i32),
        "pa_alloc_destroy": ([P], None),
        "pa_alloc_append": ([P, P, P, i32], i32),
        "pa_alloc_fork": ([P, P, i32], i32),
        "pa_alloc_writable_tail": ([P, P, P, i32, i64, i32, P, P, P], i32),
        "pa_alloc_reserve": ([P, P, P, i32, i64, i64, i32, P, P, P, i32, P], i32),
        "pa_alloc_release": ([P, P, i32], i32),
        "pa_alloc_refcount": ([P, i32], i32),
        "pa_alloc_num_free": ([P], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def status_str(status: int) -> str:
    return lib().pa_status_str(status).decode()


def _check(status: int, what: str):
    if status != PA_OK:
        msg = "%s failed: %s" % (what, status_str(status))
        if status == PA_ERR_CUDA:
            msg += " (%s)" % lib().pa_last_cuda_error().decode()
        raise PagedKVError(status, msg)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if device is not None and t.device != device:
        raise ValueError("%s must live on %s, got %s" % (name, device, t.device))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def _need_shape(t: torch.Tensor, name: str, shape):
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def _need_err(d_err: Optional[torch.Tensor], device):
    """The device error word: None, or an int32 tensor on the pool's device."""
    if d_err is not None:
        _need(d_err, "d_err", torch.int32, device)
        if d_err.numel() < 1:
            raise ValueError("d_err must hold at least one int32")


def _need_workspace(ws: Optional[torch.Tensor], device):
    if ws is not None:
        _need(ws, "workspace", None, device)


def _need_decode_args(pool, q, block_tables, context_lens, out):
    """Shapes of a decode call: q [B][H_q][D], block_tables [B][max_blocks],
    context_lens [B], out [B][H_q][D] float32 (when given)."""
    _need(q, "q", pool.io_dtype, pool.device)
    _need(block_tables, "block_tables", torch.int32, pool.device)
    _need(context_lens, "context_lens", torch.int32, pool.device)
    if q.dim() != 3 or q.shape[2] != pool.head_dim:
        raise ValueError("q must be [B][H_q][%d], got %s" % (pool.head_dim, tuple(q.shape)))
    B, Hq, D = q.shape
    if block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("block_tables must be [%d][max_blocks], got %s"
                         % (B, tuple(block_tables.shape)))
    _need_shape(context_lens, "context_lens", (B,))
    if out is not None:
        _need(out, "out", torch.float32, pool.device)
        _need_shape(out, "out", (B, Hq, D))
    return B, Hq, D


# --------------------------------------------------------------------------- pool
class KVPool:
    """K and V block pools [num_blocks][num_kv_heads][block_size][head_dim] on one device.

    dtype float32 or bfloat16 stores rows as they are; torch.float8_e4m3fn stores
    E4M3 codes (uint8 tensors k, v) with one float32 scale per row (k_scale,
    v_scale [num_blocks][num_kv_heads][block_size]); rows are then written and
    queried in bfloat16 (``io_dtype``).
    """

    def __init__(self, num_blocks: int, block_size: int, num_kv_heads: int, head_dim: int,
                 dtype: torch.dtype = torch.bfloat16, device="cuda", k=None, v=None):
        fp8 = getattr(torch, "float8_e4m3fn", None)
        if dtype not in (torch.float32, torch.bfloat16) and (fp8 is None or dtype != fp8):
            raise TypeError("pool dtype must be float32, bfloat16 or float8_e4m3fn")
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        self.num_kv_heads, self.head_dim = int(num_kv_heads), int(head_dim)
        self.dtype = dtype
        self.is_fp8 = fp8 is not None and dtype == fp8
        self.io_dtype = torch.bfloat16 if self.is_fp8 else dtype
        store = torch.uint8 if self.is_fp8 else dtype
        shape = (self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim)
        self.k = torch.empty(shape, dtype=store, device=device) if k is None else k
        self.v = torch.empty(shape, dtype=store, device=device) if v is None else v
        for t, n in ((self.k, "k"), (self.v, "v")):
            if tuple(t.shape) != shape or t.dtype != store:
                raise ValueError("pool tensor %s has the wrong shape or dtype" % n)
            _need(t, "pool." + n)
        self.device = self.k.device
        self.k_scale = self.v_scale = None
        if self.is_fp8:
            self.k_scale = torch.empty(shape[:3], dtype=torch.float32, device=self.device)
            self.v_scale = torch.empty(shape[:3], dtype=torch.float32, device=self.device)
        code = DTYPE_FP8_E4M3 if self.is_fp8 else (DTYPE_F32 if dtype == torch.float32
                                                   else DTYPE_BF16)
        self._c = pa_kv_pool(self.k.data_ptr(), self.v.data_ptr(), self.num_blocks,
                             self.block_size, self.num_kv_heads, self.head_dim, code,
                             None if self.k_scale is None else self.k_scale.data_ptr(),
                             None if self.v_scale is None else self.v_scale.data_ptr())

    @property
    def c(self):
        return ctypes.byref(self._c)

    def poison(self):
        """Fill the pools with NaN bit patterns (all bytes 0xFF; for FP8 pages the
        codes and the scales)."""
        for t in (self.k, self.v, self.k_scale, self.v_scale):
            if t is not None:
                t.view(torch.uint8).fill_(0xFF)
        return self


def page_size_bytes(pool: KVPool) -> int:
    out = ctypes.c_int64(0)
    _check(lib().pa_page_size_bytes(pool.c, ctypes.byref(out)), "pa_page_size_bytes")
    return out.value


# --------------------------------------------------------------------------- addressing
def physical_slot(table: Sequence[int], block_size: int, pos: int) -> int:
    t = np.ascontiguousarray(table, dtype=np.int32)
    out = ctypes.c_int64(0)
    _check(lib().pa_physical_slot(t.ctypes.data_as(ctypes.c_void_p), len(t), block_size, pos,
                                  ctypes.byref(out)), "pa_physical_slot")
    return out.value


def slot_mapping(table: Sequence[int], block_size: int, positions) -> np.ndarray:
    t = np.ascontiguousarray(table, dtype=np.int32)
    pos = np.ascontiguousarray(positions, dtype=np.int64)
    out = np.empty(len(pos), np.int64)
    _check(lib().pa_slot_mapping(t.ctypes.data_as(ctypes.c_void_p), len(t), block_size,
                                 pos.ctypes.data_as(ctypes.c_void_p), len(pos),
                                 out.ctypes.data_as(ctypes.c_void_p)), "pa_slot_mapping")
    return out


# --------------------------------------------------------------------------- kernels
def write_kv(pool: KVPool, k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
             d_err: Optional[torch.Tensor] = None, stream=None):
    """Scatter k_new/v_new [T][H_kv][D] into the pool at slot_mapping [T] (int64)."""
    T = int(slot_mapping.shape[0])
    _need(k_new, "k_new", pool.io_dtype, pool.device)
    _need(v_new, "v_new", pool.io_dtype, pool.device)
    _need(slot_mapping, "slot_mapping", torch.int64, pool.device)
    if tuple(k_new.shape) != (T, pool.num_kv_heads, pool.head_dim) or k_new.shape != v_new.shape:
        raise ValueError("k_new/v_new must be [T][H_kv][D] with T = len(slot_mapping)")
    _need_shape(slot_mapping, "slot_mapping", (T,))
    _need_err(d_err, pool.device)
    _check(lib().pa_write_kv(pool.c, _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), T,
                             _ptr(d_err), _stream(stream)), "pa_write_kv")


def copy_blocks(pool: KVPool, src: torch.Tensor, dst: torch.Tensor,
                d_err: Optional[torch.Tensor] = None, stream=None):
    """Block copy dst[i] <- src[i] (int32 device tensors) in both pools."""
    _need(src, "src", torch.int32, pool.device)
    _need(dst, "dst", torch.int32, pool.device)
    if src.shape != dst.shape or src.dim() != 1:
        raise ValueError("src and dst must be 1-D of equal length")
    _need_err(d_err, pool.device)
    _check(lib().pa_copy_blocks(pool.c, _ptr(src), _ptr(dst), int(src.shape[0]), _ptr(d_err),
                                _stream(stream)), "pa_copy_blocks")


def decode_partition_tokens(pool: KVPool, num_seqs: int, num_q_heads: int, max_context: int) -> int:
    out = ctypes.c_int32(0)
    _check(lib().pa_decode_partition_tokens(pool.c, num_seqs, num_q_heads, max_context,
                                            ctypes.byref(out)), "pa_decode_partition_tokens")
    return out.value


def decode_workspace_bytes(pool: KVPool, num_seqs: int, num_q_heads: int, max_context: int,
                           partition_tokens: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().pa_decode_workspace_bytes(pool.c, num_seqs, num_q_heads, max_context,
                                           partition_tokens, ctypes.byref(out)),
           "pa_decode_workspace_bytes")
    return out.value


def decode(pool: KVPool, q: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
           max_context: int, scale: float, out: Optional[torch.Tensor] = None,
           workspace: Optional[torch.Tensor] = None, partition_tokens: int = 0,
           d_err: Optional[torch.Tensor] = None, stream=None, phase: str = "all") -> torch.Tensor:
    """Paged decode attention; returns out [B][H_q][D] float32.

    phase: "all" (pa_decode), "partial" (pa_decode_partial) or "merge"
    (pa_decode_merge, which needs the workspace the partial phase filled).
    """
    B, Hq, D = _need_decode_args(pool, q, block_tables, context_lens, out)
    _need_workspace(workspace, pool.device)
    _need_err(d_err, pool.device)
    if phase not in ("all", "partial", "merge"):
        raise ValueError("phase must be 'all', 'partial' or 'merge'")
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=pool.device)
    need = decode_workspace_bytes(pool, B, Hq, max_context, partition_tokens)
    if need > 0 and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=pool.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if phase == "merge":
        _check(lib().pa_decode_merge(pool.c, Hq, _ptr(context_lens), B, int(max_context),
                                     int(partition_tokens), _ptr(out), _ptr(workspace), ws_bytes,
                                     _stream(stream)), "pa_decode_merge")
        return out
    fn = {"all": lib().pa_decode, "partial": lib().pa_decode_partial}[phase]
    _check(fn(pool.c, _ptr(q), Hq, _ptr(block_tables), int(block_tables.shape[1]),
              _ptr(context_lens), B, int(max_context), float(scale), int(partition_tokens),
              _ptr(out), _ptr(workspace), ws_bytes, _ptr(d_err), _stream(stream)),
           "pa_decode" if phase == "all" else "pa_decode_partial")
    return out


def decode_shared_workspace_bytes(pool: KVPool, num_seqs: int, num_q_heads: int,
                                  max_context: int, partition_tokens: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().pa_decode_shared_workspace_bytes(pool.c, num_seqs, num_q_heads, max_context,
                                                  partition_tokens, ctypes.byref(out)),
           "pa_decode_shared_workspace_bytes")
    return out.value


def decode_shared(pool: KVPool, q: torch.Tensor, block_tables: torch.Tensor,
                  context_lens: torch.Tensor, max_context: int, partner: torch.Tensor,
                  shared_lens: torch.Tensor, scale: float, out: Optional[torch.Tensor] = None,
                  workspace: Optional[torch.Tensor] = None, partition_tokens: int = 0,
                  d_err: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Shared-prefix-aware paged decode (pa_decode_shared); returns out [B][H_q][D].

    partner: int32 [B] (the other member of a pair, or -1); shared_lens: int32
    [B], tokens on the pair's shared leading pages.
    """
    B, Hq, D = _need_decode_args(pool, q, block_tables, context_lens, out)
    _need(partner, "partner", torch.int32, pool.device)
    _need(shared_lens, "shared_lens", torch.int32, pool.device)
    _need_shape(partner, "partner", (B,))
    _need_shape(shared_lens, "shared_lens", (B,))
    _need_workspace(workspace, pool.device)
    _need_err(d_err, pool.device)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=pool.device)
    need = decode_shared_workspace_bytes(pool, B, Hq, max_context, partition_tokens)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=pool.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pa_decode_shared(pool.c, _ptr(q), Hq, _ptr(block_tables),
                                  int(block_tables.shape[1]), _ptr(context_lens), B,
                                  int(max_context), _ptr(partner), _ptr(shared_lens),
                                  float(scale), int(partition_tokens), _ptr(out),
                                  _ptr(workspace), ws_bytes, _ptr(d_err), _stream(stream)),
           "pa_decode_shared")
    return out


def decode_window_workspace_bytes(pool: KVPool, num_seqs: int, num_q_heads: int,
                                  max_context: int, window: int, partition_tokens: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().pa_decode_window_workspace_bytes(pool.c, num_seqs, num_q_heads, max_context,
                                                  int(window), partition_tokens,
                                                  ctypes.byref(out)),
           "pa_decode_window_workspace_bytes")
    return out.value


def decode_window(pool: KVPool, q: torch.Tensor, block_tables: torch.Tensor,
                  context_lens: torch.Tensor, max_context: int, window: int, scale: float,
                  out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                  partition_tokens: int = 0, d_err: Optional[torch.Tensor] = None,
                  stream=None) -> torch.Tensor:
    """Sliding-window paged decode: the query at position n-1 attends to the last
    `window` positions; returns out [B][H_q][D] float32."""
    B, Hq, D = _need_decode_args(pool, q, block_tables, context_lens, out)
    _need_workspace(workspace, pool.device)
    _need_err(d_err, pool.device)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=pool.device)
    need = decode_window_workspace_bytes(pool, B, Hq, max_context, window, partition_tokens)
    if need > 0 and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=pool.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().pa_decode_window(pool.c, _ptr(q), Hq, _ptr(block_tables),
                                  int(block_tables.shape[1]), _ptr(context_lens), B,
                                  int(max_context), int(window), float(scale),
                                  int(partition_tokens), _ptr(out), _ptr(workspace), ws_bytes,
                                  _ptr(d_err), _stream(stream)), "pa_decode_window")
    return out


def decode_step_workspace_bytes(pool: KVPool, num_seqs: int, num_q_heads: int, max_context: int,
                                partition_tokens: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().pa_decode_step_workspace_bytes(pool.c, num_seqs, num_q_heads, max_context,
                                                partition_tokens, ctypes.byref(out)),
           "pa_decode_step_workspace_bytes")
    return out.value


def decode_step_workspace(pool: KVPool, num_seqs: int, num_q_heads: int, max_context: int,
                          partition_tokens: int = 0) -> Optional[torch.Tensor]:
    """A zero-filled workspace for decode_step (reusable for every later call of the shape)."""
    n = decode_step_workspace_bytes(pool, num_seqs, num_q_heads, max_context, partition_tokens)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=pool.device) if n > 0 else None


def decode_step(pool: KVPool, k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                q: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                max_context: int, scale: float, workspace: Optional[torch.Tensor],
                out: Optional[torch.Tensor] = None, partition_tokens: int = 0,
                d_err: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """pa_decode_step: write each sequence's new token and attend, in one launch.

    workspace comes from decode_step_workspace() (zero-filled once, then reused).
    """
    _need(k_new, "k_new", pool.io_dtype, pool.device)
    _need(v_new, "v_new", pool.io_dtype, pool.device)
    _need(slot_mapping, "slot_mapping", torch.int64, pool.device)
    B, Hq, D = _need_decode_args(pool, q, block_tables, context_lens, out)
    if tuple(k_new.shape) != (B, pool.num_kv_heads, pool.head_dim) or k_new.shape != v_new.shape:
        raise ValueError("k_new/v_new must be [B][H_kv][D]")
    if tuple(slot_mapping.shape) != (B,):
        raise ValueError("slot_mapping must be [B]")
    _need_workspace(workspace, pool.device)
    _need_err(d_err, pool.device)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=pool.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().pa_decode_step(pool.c, _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(q), Hq,
                                _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens),
                                B, int(max_context), float(scale), int(partition_tokens), _ptr(out),
                                _ptr(workspace), ws_bytes, _ptr(d_err), _stream(stream)),
           "pa_decode_step")
    return out


def prefill(pool: KVPool, q: torch.Tensor, cu_seqlens_q: torch.Tensor, context_lens: torch.Tensor,
            block_tables: torch.Tensor, max_q_len: int, max_context: int, scale: float,
            causal: bool = True, out: Optional[torch.Tensor] = None,
            d_err: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Paged chunked-prefill attention; returns out [T][H_q][D] float32."""
    _need(q, "q", pool.io_dtype, pool.device)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, pool.device)
    _need(context_lens, "context_lens", torch.int32, pool.device)
    _need(block_tables, "block_tables", torch.int32, pool.device)
    if q.dim() != 3 or q.shape[2] != pool.head_dim:
        raise ValueError("q must be [T][H_q][%d], got %s" % (pool.head_dim, tuple(q.shape)))
    T, Hq, D = q.shape
    B = int(context_lens.shape[0]) if context_lens.dim() == 1 else -1
    if B < 0:
        raise ValueError("context_lens must be 1-D")
    _need_shape(cu_seqlens_q, "cu_seqlens_q", (B + 1,))
    if block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("block_tables must be [%d][max_blocks], got %s"
                         % (B, tuple(block_tables.shape)))
    _need_err(d_err, pool.device)
    if out is None:
        out = torch.empty((T, Hq, D), dtype=torch.float32, device=pool.device)
    _need(out, "out", torch.float32, pool.device)
    _need_shape(out, "out", (T, Hq, D))
    _check(lib().pa_prefill(pool.c, _ptr(q), T, Hq, _ptr(cu_seqlens_q), _ptr(context_lens),
                            _ptr(block_tables), int(block_tables.shape[1]),
                            int(context_lens.shape[0]), int(max_q_len), int(max_context),
                            float(scale), 1 if causal else 0, _ptr(out), _ptr(d_err),
                            _stream(stream)), "pa_prefill")
    return out


# --------------------------------------------------------------------------- allocator
class BlockTable:
    """One sequence's block table: an int32 host buffer with room to grow."""

    def __init__(self, capacity: int = 64, ids: Optional[Sequence[int]] = None):
        ids = [] if ids is None else list(ids)
        self.buf = np.full(max(int(capacity), len(ids), 1), -1, dtype=np.int32)
        self.buf[:len(ids)] = ids
        self.n = ctypes.c_int32(len(ids))

    def __len__(self):
        return self.n.value

    def ids(self) -> np.ndarray:
        return self.buf[:self.n.value]

    def tolist(self) -> list:
        return [int(x) for x in self.ids()]

    def reserve(self, extra: int):
        need = self.n.value + int(extra)
        if need > len(self.buf):
            nb = np.full(max(need, 2 * len(self.buf)), -1, dtype=np.int32)
            nb[:self.n.value] = self.ids()
            self.buf = nb

    @property
    def ptr(self):
        return self.buf.ctypes.data_as(ctypes.c_void_p)


class Allocator:
    """Host block allocator (refcounts, LIFO free list, fork, copy-on-write tail)."""

    def __init__(self, num_blocks: int, free_order: Optional[Sequence[int]] = None):
        self._h = ctypes.c_void_p()
        fo = None
        if free_order is not None:
            self._fo = np.ascontiguousarray(free_order, dtype=np.int32)
            fo = self._fo.ctypes.data_as(ctypes.c_void_p)
        _check(lib().pa_alloc_create(int(num_blocks), fo, ctypes.byref(self._h)), "pa_alloc_create")
        self.num_blocks = int(num_blocks)

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value and _lib is not None:
            _lib.pa_alloc_destroy(self._h)
            self._h = ctypes.c_void_p()

    def append(self, t: BlockTable) -> int:
        t.reserve(1)
        _check(lib().pa_alloc_append(self._h, t.ptr, ctypes.byref(t.n), len(t.buf)),
               "pa_alloc_append")
        return int(t.buf[t.n.value - 1])

    def fork(self, t: BlockTable) -> BlockTable:
        _check(lib().pa_alloc_fork(self._h, t.ptr, len(t)), "pa_alloc_fork")
        return BlockTable(len(t.buf), t.ids())

    def writable_tail(self, t: BlockTable, logical_length: int, block_size: int):
        """(block, offset, cow_src) for the token at ``logical_length``; updates ``t``."""
        t.reserve(1)
        blk, off, cow = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _check(lib().pa_alloc_writable_tail(self._h, t.ptr, ctypes.byref(t.n), len(t.buf),
                                            int(logical_length), int(block_size),
                                            ctypes.byref(blk), ctypes.byref(off),
                                            ctypes.byref(cow)), "pa_alloc_writable_tail")
        return blk.value, off.value, cow.value

    def reserve(self, t: BlockTable, logical_length: int, count: int, block_size: int):
        """Slots (int64 [count]) and copy-on-write pairs for positions
        [logical_length, logical_length + count)."""
        t.reserve(count // block_size + 2)
        slots = np.empty(int(count), np.int64)
        cap = count // block_size + 2
        src = np.empty(cap, np.int32)
        dst = np.empty(cap, np.int32)
        n_cow = ctypes.c_int32(0)
        _check(lib().pa_alloc_reserve(self._h, t.ptr, ctypes.byref(t.n), len(t.buf),
                                      int(logical_length), int(count), int(block_size),
                                      slots.ctypes.data_as(ctypes.c_void_p),
                                      src.ctypes.data_as(ctypes.c_void_p),
                                      dst.ctypes.data_as(ctypes.c_void_p), cap,
                                      ctypes.byref(n_cow)), "pa_alloc_reserve")
        return slots, list(zip(src[:n_cow.value].tolist(), dst[:n_cow.value].tolist()))

    def release(self, t: BlockTable):
        _check(lib().pa_alloc_release(self._h, t.ptr, len(t)), "pa_alloc_release")
        t.n.value = 0

    def refcount(self, block: int) -> int:
        return int(lib().pa_alloc_refcount(self._h, int(block)))

    def num_free(self) -> int:
        return int(lib().pa_alloc_num_free(self._h))


def pack_tables(tables, width: Optional[int] = None, device="cuda") -> torch.Tensor:
    """Block tables (BlockTable or id lists) as a padded int32 [B][width] tensor (pad -1)."""
    ids = [t.ids() if isinstance(t, BlockTable) else np.asarray(t, np.int32) for t in tables]
    w = max(1, max((len(t) for t in ids), default=1)) if width is None else int(width)
    arr = np.full((len(ids), w), -1, dtype=np.int32)
    for i, t in enumerate(ids):
        arr[i, :len(t)] = t
    return torch.from_numpy(arr).to(device)

"""Float64 CPU oracle for the paged KV-cache attention path.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library: it does its own slot arithmetic, its own allocator
bookkeeping, its own pool writes and copies, and its own attention in float64
(``attention.c``).  It is slow and plain on purpose.

Sources (page title, section):
  P1 = "03｜PagedAttention 与 KV Cache 内存系统" (llm-infra-atlas.github.io)
  P2 = "KV Cache：容量、布局与生命周期" (wineandchord.com)
  P3 = "PagedAttention 的原理是什么？它如何降低 KV Cache 的内存浪费？" (offer.aigcbaba.com)
  P4 = "vLLM学习笔记-显存管理之PagedAttention" (amentiraz.github.io)

Pins (tests/test_oracle.py, tests/test_oracle_fp8.py): the worked examples
of P2 "Page-table 寻址" and P2 "引用计数与尾块 COW" (tests/golden/), the
out-of-range failure, refcount and copy-on-write invariants (P2 "生命周期与所有权"),
paged == contiguous bit identity (P1 §4, P3 §五), brute force against a
library softmax-attention routine on tiny inputs, closed forms (one key,
identical keys, a dominant key), split/merge equivalence (also with partition
maxima 1000 apart), causal-row == truncated-decode identity, and GQA head
mapping.  tests/test_oracle_mutations.py plants mistakes in a copy of this
package and checks that each one fails a pin.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None


# --------------------------------------------------------------------------- build / load
def build(force: bool = False) -> str:
    """Compile attention.c into liboracle.so (plain gcc, OpenMP, no fast-math)."""
    src = os.path.join(_HERE, "attention.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               src, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.orc_physical_slot.argtypes = [P, i64, i64, i64, P]
        lib.orc_decode.argtypes = [P, P, ctypes.c_int, i32, i32, i32, i32, P, i32, P, i32, P, i32,
                                   f64, P, i32, P]
        lib.orc_decode_window.argtypes = [P, P, ctypes.c_int, i32, i32, i32, i32, P, i32, P,
                                          i32, P, i32, i32, f64, P, i32, P]
        lib.orc_decode_contiguous.argtypes = [P, P, ctypes.c_int, i32, i32, i32, P, i32, P, i32,
                                              f64, P]
        lib.orc_decode_split.argtypes = [P, P, ctypes.c_int, i32, i32, i32, i32, P, i32, P, i32,
                                         P, i32, f64, i32, P]
        lib.orc_prefill.argtypes = [P, P, ctypes.c_int, i32, i32, i32, i32, P, i32, P, P, P, i32,
                                    i32, f64, i32, P, i32, P]
        lib.orc_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().orc_num_threads())


class OracleError(RuntimeError):
    pass


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int):
    if rc == -2:
        raise IndexError("logical block is not allocated or block id is outside the pool")
    if rc == -3:
        raise ValueError("physical block id must be non-negative")
    if rc != 0:
        raise ValueError("invalid argument (oracle rc=%d)" % rc)


# --------------------------------------------------------------------------- addressing
def physical_slot(block_table: Sequence[int], block_size: int, token_pos: int) -> int:
    """Slot of a token position through a block table (P2 "Page-table 寻址", P1 §3).

    The logical block is pos // B_p and the offset pos mod B_p; the slot is
    table[logical] * B_p + offset.  A non-positive block size or negative
    position is a ValueError, a logical block past the table an IndexError, a
    negative physical id a ValueError.
    """
    if block_size <= 0 or token_pos < 0:
        raise ValueError("block size must be positive and position non-negative")
    logical = token_pos // block_size
    offset = token_pos - logical * block_size
    if logical >= len(block_table):
        raise IndexError("logical block %d is not allocated" % logical)
    phys = int(block_table[logical])
    if phys < 0:
        raise ValueError("physical block id must be non-negative")
    return phys * block_size + offset


def physical_slot_c(block_table: Sequence[int], block_size: int, token_pos: int) -> int:
    """The same through attention.c (so both oracle halves are pinned alike)."""
    t = np.ascontiguousarray(block_table, dtype=np.int32)
    out = np.zeros(1, np.int64)
    _check(_load().orc_physical_slot(_ptr(t), len(t), block_size, token_pos, _ptr(out)))
    return int(out[0])


# --------------------------------------------------------------------------- ownership
class BlockPool:
    """Block ownership of P2 "引用计数与尾块 COW" and "生命周期与所有权".

    ``refcount[b]`` counts the logical sequences holding block b; the free list
    is a Python list and allocation pops from its end (the pages' ``pop()``);
    a freed block goes back on the end, so it is the next one reused (P1 §5:
    blocks without a prefix hash are reused first).
    """

    def __init__(self, num_blocks: int, free_order: Optional[Sequence[int]] = None):
        self.num_blocks = num_blocks
        self.refcount = [0] * num_blocks
        self.free = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]

    def _pop(self) -> int:
        if not self.free:
            raise MemoryError("no free block")
        return self.free.pop()

    def append(self, table: list) -> int:
        """Give ``table`` one more logical block, exclusively owned (ref 1)."""
        b = self._pop()
        self.refcount[b] = 1
        table.append(b)
        return b

    def fork(self, table: list) -> list:
        """A child table naming the same blocks; each block gains a holder."""
        child = list(table)
        for b in child:
            self.refcount[b] += 1
        return child

    def writable_tail(self, table: list, logical_length: int, block_size: int):
        """Where the token at position ``logical_length`` may be written.

        Returns (block, offset, cow_src).  Offset 0 starts a new logical block,
        which is appended (the table must then hold exactly logical_length /
        block_size entries).  A partially filled block with more than one
        holder is replaced by a fresh exclusive block and ``cow_src`` names the
        old one, whose committed rows the caller must copy before publishing
        the table; otherwise cow_src is -1.
        """
        if block_size <= 0 or logical_length < 0:
            raise ValueError("invalid block size or length")
        logical, offset = divmod(logical_length, block_size)
        cow_src = -1
        if offset == 0:
            if logical != len(table):
                raise ValueError("next block must be appended at the end of the table")
            self.append(table)
        else:
            if logical >= len(table):
                raise IndexError("logical block is not allocated")
            cur = table[logical]
            if self.refcount[cur] > 1:
                fresh = self._pop()
                self.refcount[cur] -= 1
                self.refcount[fresh] = 1
                table[logical] = fresh
                cow_src = cur
        return table[logical], offset, cow_src

    def release(self, table: list):
        """Drop one holder from every block of ``table``; free blocks at zero."""
        for b in table:
            if self.refcount[b] <= 0:
                raise ValueError("refcount underflow on block %d" % b)
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self.free.append(b)
        table.clear()


# --------------------------------------------------------------------------- pool storage
def poisoned_pool(num_blocks: int, num_kv_heads: int, block_size: int, head_dim: int, dtype: str):
    """K and V pools [N][H_kv][B_p][D] filled with NaN bit patterns (all ones)."""
    npdt = np.float32 if dtype == "f32" else np.uint16
    shape = (num_blocks, num_kv_heads, block_size, head_dim)
    k = np.empty(shape, dtype=npdt)
    v = np.empty(shape, dtype=npdt)
    k.view(np.uint8)[...] = 0xFF
    v.view(np.uint8)[...] = 0xFF
    return k, v


def write_kv(kpool: np.ndarray, vpool: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
             slot_mapping: Sequence[int]):
    """Scatter one K and one V row per token into its slot (P1 §4.1).

    Exactly len(slot_mapping) tokens are written: row t goes to block
    slot // B_p at offset slot mod B_p, for every KV head.
    """
    N, H, Bp, D = kpool.shape
    for t, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot < 0 or slot >= N * Bp:
            raise IndexError("slot %d outside the pool" % slot)
        blk, off = divmod(slot, Bp)
        kpool[blk, :, off, :] = k_new[t]
        vpool[blk, :, off, :] = v_new[t]


def copy_blocks(kpool: np.ndarray, vpool: np.ndarray, src: Sequence[int], dst: Sequence[int]):
    """Whole-block copy dst <- src for K and V, all heads (P1 §5 copy-on-write)."""
    N = kpool.shape[0]
    for a, b in zip(src, dst):
        if not (0 <= a < N and 0 <= b < N):
            raise IndexError("block id outside the pool")
        kpool[b] = kpool[a]
        vpool[b] = vpool[a]


def _dtype_code(arr: np.ndarray) -> int:
    if arr.dtype == np.float32:
        return 0
    if arr.dtype == np.uint16:
        return 1
    if arr.dtype == np.float64:
        return 2
    raise TypeError("pool/query arrays must be float32, uint16 (bf16 bits) or float64")


def _tables_array(tables) -> np.ndarray:
    width = max(1, max((len(t) for t in tables), default=1))
    arr = np.full((len(tables), width), -1, dtype=np.int32)
    for i, t in enumerate(tables):
        arr[i, :len(t)] = t
    return arr


def decode(kpool, vpool, q, tables, context_lens, scale, rows=None) -> np.ndarray:
    """Decode attention in float64 (see attention.c: orc_decode).

    q: [B][H_q][D] in the pool's dtype; tables: list of block lists;
    context_lens: tokens visible to each query, the new one included.
    rows: optional [(s, g)] list; the result then has one row per pair.
    """
    lib = _load()
    N, H, Bp, D = kpool.shape
    q = np.ascontiguousarray(q)
    B, Hq, _ = q.shape
    tab = _tables_array(tables)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    if rows is None:
        out = np.zeros((B, Hq, D), np.float64)
        r_arr, n_rows = None, 0
    else:
        r_arr = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 2)
        n_rows = r_arr.shape[0]
        out = np.zeros((n_rows, D), np.float64)
    rc = lib.orc_decode(_ptr(kpool), _ptr(vpool), _dtype_code(kpool), N, Bp, H, D, _ptr(q), Hq,
                        _ptr(tab), tab.shape[1], _ptr(lens), B, float(scale),
                        None if r_arr is None else _ptr(r_arr), n_rows, _ptr(out))
    _check(rc)
    return out


def decode_window(kpool, vpool, q, tables, context_lens, scale, window, rows=None) -> np.ndarray:
    """Sliding-window decode in float64 (see attention.c: orc_decode_window): the
    query at position n - 1 attends to positions max(0, n - window) .. n - 1;
    window <= 0 means the whole context."""
    lib = _load()
    N, H, Bp, D = kpool.shape
    q = np.ascontiguousarray(q)
    B, Hq, _ = q.shape
    tab = _tables_array(tables)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    if rows is None:
        out = np.zeros((B, Hq, D), np.float64)
        r_arr, n_rows = None, 0
    else:
        r_arr = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 2)
        n_rows = r_arr.shape[0]
        out = np.zeros((n_rows, D), np.float64)
    rc = lib.orc_decode_window(_ptr(kpool), _ptr(vpool), _dtype_code(kpool), N, Bp, H, D,
                               _ptr(q), Hq, _ptr(tab), tab.shape[1], _ptr(lens), B, int(window),
                               float(scale), None if r_arr is None else _ptr(r_arr), n_rows,
                               _ptr(out))
    _check(rc)
    return out


def decode_contiguous(kcache, vcache, q, context_lens, scale) -> np.ndarray:
    """Decode over the contiguous P4 layout cache[B][max_seq][H_kv][D]."""
    lib = _load()
    B, max_seq, H, D = kcache.shape
    q = np.ascontiguousarray(q)
    Hq = q.shape[1]
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.zeros((B, Hq, D), np.float64)
    _check(lib.orc_decode_contiguous(_ptr(np.ascontiguousarray(kcache)),
                                     _ptr(np.ascontiguousarray(vcache)), _dtype_code(kcache),
                                     max_seq, H, D, _ptr(q), Hq, _ptr(lens), B, float(scale),
                                     _ptr(out)))
    return out


def decode_split(kpool, vpool, q, tables, context_lens, scale, part_tokens) -> np.ndarray:
    """Decode through per-partition (max, exp_sum, weighted V) states and a merge."""
    lib = _load()
    N, H, Bp, D = kpool.shape
    q = np.ascontiguousarray(q)
    B, Hq, _ = q.shape
    tab = _tables_array(tables)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.zeros((B, Hq, D), np.float64)
    _check(lib.orc_decode_split(_ptr(kpool), _ptr(vpool), _dtype_code(kpool), N, Bp, H, D, _ptr(q),
                                Hq, _ptr(tab), tab.shape[1], _ptr(lens), B, float(scale),
                                int(part_tokens), _ptr(out)))
    return out


def prefill(kpool, vpool, q, cu_seqlens_q, context_lens, tables, scale, causal=True,
            rows=None) -> np.ndarray:
    """Chunked-prefill attention in float64 (see attention.c: orc_prefill).

    q: [T][H_q][D]; cu_seqlens_q: [B+1]; context_lens: cache tokens per
    sequence including the new ones.  rows: optional [(token, q-head)] list.
    """
    lib = _load()
    N, H, Bp, D = kpool.shape
    q = np.ascontiguousarray(q)
    T, Hq, _ = q.shape
    tab = _tables_array(tables)
    cu = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    B = len(lens)
    if rows is None:
        out = np.zeros((T, Hq, D), np.float64)
        r_arr, n_rows = None, 0
    else:
        r_arr = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 2)
        n_rows = r_arr.shape[0]
        out = np.zeros((n_rows, D), np.float64)
    _check(lib.orc_prefill(_ptr(kpool), _ptr(vpool), _dtype_code(kpool), N, Bp, H, D, _ptr(q), Hq,
                           _ptr(cu), _ptr(lens), _ptr(tab), tab.shape[1], B, float(scale),
                           1 if causal else 0, None if r_arr is None else _ptr(r_arr), n_rows,
                           _ptr(out)))
    return out


# --------------------------------------------------------------------------- scenario
def to_numpy_bits(t) -> np.ndarray:
    """torch tensor (f32 or bf16) -> numpy float32 or uint16 bit pattern array."""
    import torch
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact float64 values of f32 or bf16-bit arrays."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


class OracleCache:
    """The oracle's own view of a workload after its tokens are written.

    Builds tables with ``BlockPool`` in sequence order, runs the shared-prefix
    scenario (parent writes the prefix, fork, each member goes through
    ``writable_tail`` and copies the tail on copy-on-write), writes every
    cached token and then this step's new tokens through ``write_kv``.
    ``events`` records the allocator decisions so the product's allocator can
    be compared against them.
    """

    def __init__(self, wl, write_new: bool = True):
        self.wl = wl
        self.pool = BlockPool(wl.num_blocks, wl.free_order)
        self.k, self.v = poisoned_pool(wl.num_blocks, wl.num_kv_heads, wl.block_size,
                                       wl.head_dim, wl.dtype)
        self.tables = [[] for _ in range(wl.num_seqs)]
        self.cow_pairs = []
        Bp = wl.block_size
        done = set()
        for s in range(wl.num_seqs):
            if s in done:
                continue
            partner = -1 if wl.pair_of is None else int(wl.pair_of[s])
            if partner >= 0:
                P = int(wl.prefix_len[s])
                parent = []
                self._write_range(s, parent, 0, P)
                members = sorted([s, partner])
                self.tables[members[0]] = parent
                self.tables[members[1]] = self.pool.fork(parent)
                for m in members:
                    self._write_range(m, self.tables[m], P, int(wl.cached_lens[m]))
                done.update(members)
            else:
                self._write_range(s, self.tables[s], 0, int(wl.cached_lens[s]))
                done.add(s)
        if write_new:
            self.write_new()

    def _write_range(self, s, table, start, end):
        """Commit tokens [start, end) of sequence s, allocating as the pages do."""
        wl, Bp = self.wl, self.wl.block_size
        if end <= start:
            return
        k, v = wl.kv_values(s, start, end)
        k, v = to_numpy_bits(k), to_numpy_bits(v)
        slots = []
        for pos in range(start, end):
            blk, off, cow = self.pool.writable_tail(table, pos, Bp)
            if cow >= 0:
                copy_blocks(self.k, self.v, [cow], [blk])
                self.cow_pairs.append((cow, blk))
            slots.append(blk * Bp + off)
        write_kv(self.k, self.v, k, v, slots)

    def write_new(self):
        wl = self.wl
        for s in range(wl.num_seqs):
            c, n = int(wl.cached_lens[s]), int(wl.new_lens[s])
            self._write_range(s, self.tables[s], c, c + n)

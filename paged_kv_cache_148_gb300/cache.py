"""Host-side owner of a paged KV pool.

``PagedCache`` keeps one block table per sequence, asks the C allocator for
blocks (``pa_alloc_reserve``: the copy-on-write tail rule of "KV Cache：容量、
布局与生命周期", section 引用计数与尾块 COW) and commits tokens on the device in
the order that rule requires: first ``pa_copy_blocks`` for every copy-on-write
decision, then ``pa_write_kv`` of the tokens ("03｜PagedAttention 与 KV Cache
内存系统" §4.1 write path).  All device work goes through the C ABI.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np
import torch

from . import Allocator, BlockTable, KVPool, copy_blocks, pack_tables, write_kv


class PagedCache:
    def __init__(self, num_blocks: int, block_size: int, num_kv_heads: int, head_dim: int,
                 dtype: torch.dtype = torch.bfloat16, device="cuda",
                 free_order: Optional[Sequence[int]] = None, poison: bool = True):
        self.pool = KVPool(num_blocks, block_size, num_kv_heads, head_dim, dtype, device)
        if poison:
            self.pool.poison()
        self.alloc = Allocator(num_blocks, free_order)
        self.block_size = int(block_size)
        self.tables: List[BlockTable] = []
        self.lengths: List[int] = []
        self.device = self.pool.device

    # ---------------------------------------------------------------- sequences
    def add_sequence(self) -> int:
        self.tables.append(BlockTable())
        self.lengths.append(0)
        return len(self.tables) - 1

    def fork(self, sid: int) -> int:
        """A new sequence sharing every block of ``sid`` (one more holder each)."""
        self.tables.append(self.alloc.fork(self.tables[sid]))
        self.lengths.append(self.lengths[sid])
        return len(self.tables) - 1

    def release(self, sid: int):
        self.alloc.release(self.tables[sid])
        self.lengths[sid] = 0

    # ---------------------------------------------------------------- tokens
    def reserve(self, sid: int, count: int):
        """Allocate positions for ``count`` new tokens; returns (slots, cow_pairs)."""
        slots, cows = self.alloc.reserve(self.tables[sid], self.lengths[sid], count,
                                         self.block_size)
        self.lengths[sid] += int(count)
        return slots, cows

    def commit(self, slots, k: torch.Tensor, v: torch.Tensor, cows=(), d_err=None, stream=None):
        """Copy-on-write copies (if any), then the scatter write of k/v rows."""
        if len(cows):
            src = torch.tensor([a for a, _ in cows], dtype=torch.int32).to(self.device)
            dst = torch.tensor([b for _, b in cows], dtype=torch.int32).to(self.device)
            copy_blocks(self.pool, src, dst, d_err=d_err, stream=stream)
        if len(slots):
            sm = slots if isinstance(slots, torch.Tensor) else torch.from_numpy(np.asarray(slots, np.int64))
            write_kv(self.pool, k, v, sm.to(self.device), d_err=d_err, stream=stream)

    def append(self, sid: int, k: torch.Tensor, v: torch.Tensor, d_err=None, stream=None):
        slots, cows = self.reserve(sid, int(k.shape[0]))
        self.commit(slots, k.to(self.device), v.to(self.device), cows, d_err, stream)
        return slots, cows

    # ---------------------------------------------------------------- metadata
    def block_tables(self, sids: Optional[Sequence[int]] = None, width: Optional[int] = None):
        sids = range(len(self.tables)) if sids is None else sids
        return pack_tables([self.tables[s] for s in sids], width, self.device)

    def context_lens(self, sids: Optional[Sequence[int]] = None):
        sids = range(len(self.tables)) if sids is None else sids
        return torch.tensor([self.lengths[s] for s in sids], dtype=torch.int32).to(self.device)

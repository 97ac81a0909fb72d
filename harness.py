"""Materialise a seeded workload on the GPU through the library's public API.

Used by the GPU tests, ``bench.py`` and ``__graft_entry__.smoke()``.  The
allocation order matches the oracle's (``oracle.OracleCache``): sequences in
index order, a shared-prefix pair as parent prefix -> fork -> each member's
private tokens, then this step's new tokens for every sequence.  All device
work goes through the library (pa_alloc_reserve, pa_copy_blocks,
pa_write_kv); nothing here computes a result.
"""
from __future__ import annotations

import numpy as np
import torch

from paged_kv_cache_148_gb300 import (decode, decode_step, decode_step_workspace, decode_window,
                                      decode_window_workspace_bytes, decode_workspace_bytes,
                                      prefill, write_kv)
from paged_kv_cache_148_gb300.cache import PagedCache

WRITE_CHUNK = 32768  # tokens per host->device batch while filling the cache


class GpuWorkload:
    def __init__(self, wl, device="cuda", reserve_new: bool = True):
        self.wl = wl
        self.device = torch.device(device)
        self.cache = PagedCache(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim,
                                wl.pool_torch_dtype, self.device, wl.free_order)
        self.sid = [None] * wl.num_seqs
        self.cow_pairs = []
        done = set()
        for s in range(wl.num_seqs):
            if s in done:
                continue
            partner = -1 if wl.pair_of is None else int(wl.pair_of[s])
            if partner >= 0:
                P = int(wl.prefix_len[s])
                members = sorted([s, partner])
                parent = self.cache.add_sequence()
                self._fill(members[0], parent, 0, P)
                self.sid[members[0]] = parent
                self.sid[members[1]] = self.cache.fork(parent)
                for m in members:
                    self._fill(m, self.sid[m], P, int(wl.cached_lens[m]))
                done.update(members)
            else:
                self.sid[s] = self.cache.add_sequence()
                self._fill(s, self.sid[s], 0, int(wl.cached_lens[s]))
                done.add(s)
        if reserve_new:
            self.reserve_new()

    def _fill(self, s, sid, start, end):
        if end <= start:
            return
        slots, cows = self.cache.reserve(sid, end - start)
        self.cow_pairs += cows
        self.cache.commit([], None, None, cows)
        for a in range(start, end, WRITE_CHUNK):
            b = min(end, a + WRITE_CHUNK)
            k, v = self.wl.kv_values(s, a, b)
            self.cache.commit(slots[a - start:b - start], k.to(self.device), v.to(self.device))

    # ------------------------------------------------------------------ the step
    def reserve_new(self):
        """Host-side scheduling of this step's tokens: slots, COW copies, inputs."""
        wl = self.wl
        slots = []
        for s in range(wl.num_seqs):
            sl, cows = self.cache.reserve(self.sid[s], int(wl.new_lens[s]))
            self.cow_pairs += cows
            self.cache.commit([], None, None, cows)
            slots.append(sl)
        self.slot_mapping_host = np.concatenate(slots).astype(np.int64)
        self.slot_mapping = torch.from_numpy(self.slot_mapping_host).to(self.device)
        k_new, v_new = wl.new_kv()
        self.k_new_host, self.v_new_host = k_new, v_new
        self.q_host = wl.queries()
        self.k_new = k_new.to(self.device)
        self.v_new = v_new.to(self.device)
        self.q = self.q_host.to(self.device)
        self.block_tables = self.cache.block_tables(self.sid)
        self.context_lens = self.cache.context_lens(self.sid)
        self.max_context = int(wl.total_lens.max())
        self.max_q = int(wl.new_lens.max())
        self.cu_seqlens_q = torch.from_numpy(
            np.concatenate([[0], np.cumsum(wl.new_lens)]).astype(np.int32)).to(self.device)
        self.err = torch.zeros(1, dtype=torch.int32, device=self.device)
        if wl.kind == "decode":
            self.out = torch.empty((wl.num_seqs, wl.num_q_heads, wl.head_dim), dtype=torch.float32,
                                   device=self.device)
        else:
            self.out = torch.empty((int(wl.new_lens.sum()), wl.num_q_heads, wl.head_dim),
                                   dtype=torch.float32, device=self.device)
        self.partition_tokens = 0
        self.window = 0  # decode: sliding window in positions (0 = the whole context)
        self._alloc_workspace()

    def _alloc_workspace(self):
        if self.wl.kind != "decode":
            self.workspace = self.step_workspace = None
            return
        if self.window > 0:
            nb = decode_window_workspace_bytes(self.cache.pool, self.wl.num_seqs,
                                               self.wl.num_q_heads, self.max_context, self.window,
                                               self.partition_tokens)
        else:
            nb = decode_workspace_bytes(self.cache.pool, self.wl.num_seqs, self.wl.num_q_heads,
                                        self.max_context, self.partition_tokens)
        self.workspace = torch.empty(max(nb, 16), dtype=torch.uint8, device=self.device)
        # pa_decode_step: zero-filled once, its semaphores return to zero every call
        self.step_workspace = decode_step_workspace(self.cache.pool, self.wl.num_seqs,
                                                    self.wl.num_q_heads, self.max_context,
                                                    self.partition_tokens)

    def set_partition_tokens(self, n: int):
        self.partition_tokens = int(n)
        self._alloc_workspace()

    def set_window(self, w: int):
        """Decode attends only to the last w positions (pa_decode_window); 0 = all."""
        self.window = int(w)
        self._alloc_workspace()

    def write_new(self, stream=None):
        write_kv(self.cache.pool, self.k_new, self.v_new, self.slot_mapping, d_err=self.err,
                 stream=stream)

    def attend(self, stream=None, phase: str = "all"):
        wl = self.wl
        if wl.kind == "decode" and self.window > 0:
            if phase != "all":
                raise ValueError("a windowed decode runs as one call")
            return decode_window(self.cache.pool, self.q, self.block_tables, self.context_lens,
                                 self.max_context, self.window, wl.scale, out=self.out,
                                 workspace=self.workspace, partition_tokens=self.partition_tokens,
                                 d_err=self.err, stream=stream)
        if wl.kind == "decode":
            return decode(self.cache.pool, self.q, self.block_tables, self.context_lens,
                          self.max_context, wl.scale, out=self.out, workspace=self.workspace,
                          partition_tokens=self.partition_tokens, d_err=self.err, stream=stream,
                          phase=phase)
        return prefill(self.cache.pool, self.q, self.cu_seqlens_q, self.context_lens,
                       self.block_tables, self.max_q, self.max_context, wl.scale,
                       causal=wl.causal, out=self.out, d_err=self.err, stream=stream)

    def attend_fused(self, stream=None):
        """Decode only: this step's new token written and attended in one launch."""
        wl = self.wl
        return decode_step(self.cache.pool, self.k_new, self.v_new, self.slot_mapping, self.q,
                           self.block_tables, self.context_lens, self.max_context, wl.scale,
                           self.step_workspace, out=self.out,
                           partition_tokens=self.partition_tokens, d_err=self.err, stream=stream)

    def step(self, stream=None, fused: bool = False):
        """One pass of the hot path: scatter this step's K/V, then attention
        (for decode with fused=True: both in pa_decode_step's single launch)."""
        if fused and self.wl.kind == "decode":
            return self.attend_fused(stream)
        self.write_new(stream)
        return self.attend(stream)

    def tables_list(self):
        return [self.cache.tables[self.sid[s]].tolist() for s in range(self.wl.num_seqs)]

    def max_parts(self) -> int:
        if self.wl.kind != "decode":
            return 1
        from paged_kv_cache_148_gb300 import decode_partition_tokens
        pt = self.partition_tokens or decode_partition_tokens(
            self.cache.pool, self.wl.num_seqs, self.wl.num_q_heads, self.max_context)
        return -(-self.max_context // pt)

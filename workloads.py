"""Seeded synthetic inputs for the paged-attention workloads.

This module only draws numbers: context lengths, the order in which the
physical block pool hands out free blocks, and the K/V/Q values. It holds none
of the method's arithmetic (no slot computation, no attention, no allocation
policy), so the CUDA path and the oracle can both consume it without sharing
any code that computes a result.

Workload recipes (sizes, distributions, seeds):

* Structure uses ``numpy.random.default_rng(1000 + k)`` and values use a torch
  CPU generator seeded with ``2000 + k`` for workload ``k`` (1..5). Values are
  drawn as float32 N(0, 1) and rounded to the storage dtype (bf16 rounding is
  round-to-nearest-even, done by ``torch.Tensor.to``).
* ``decode_tiny``      (k=1): 4 seqs, cached length U[1, 64], H_q=4, H_kv=2,
  D=64, block size 4, fp32, 128 physical blocks.
* ``decode_gqa``       (k=2): 64 seqs, U[128, 4096], H_q=32, H_kv=8, D=128,
  block size 16, bf16, pool = 1.5x the blocks the batch needs.
* ``decode_mha``       (k=3): 256 seqs, lognormal(ln 512, 1.0) clipped to
  [16, 2048], H_q=H_kv=32, D=128, block size 16, bf16.
* ``decode_long_shared`` (k=4): 8 seqs in 4 pairs, U[32768, 131072],
  H_q=64, H_kv=8, D=128, block size 16, bf16; each pair shares a prefix of
  floor(0.75 * min(L_a, L_b)) tokens, moved one token down when it would fall
  on a block boundary so that the shared tail block is partially filled.
* ``prefill``          (k=5): 16 seqs, 2048 cached + 512 new tokens each,
  H_q=32, H_kv=8, D=128, block size 16, bf16, causal.

Every workload also has a ``scale`` that shrinks it (fewer sequences, shorter
contexts) for tests the float64 oracle must finish in seconds.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch


@dataclasses.dataclass
class Workload:
    name: str
    kind: str                 # "decode" or "prefill"
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str                # "f32" or "bf16" (storage and operand type)
    scale: float              # softmax scale, 1/sqrt(head_dim)
    cached_lens: np.ndarray   # int64 [B]: tokens already in the cache, positions 0..c-1
    new_lens: np.ndarray      # int64 [B]: tokens written this step (1 for decode)
    num_blocks: int           # physical blocks in the pool
    free_order: np.ndarray    # int32 [num_blocks]: the free list; allocation pops from the END
    causal: bool = True
    # shared-prefix structure: pair_of[s] = partner index or -1; prefix_len[s] = shared tokens
    pair_of: Optional[np.ndarray] = None
    prefix_len: Optional[np.ndarray] = None
    seed_values: int = 0
    # "native": the pool stores rows in `dtype`; "fp8": E4M3 codes with one float32
    # scale per (token, kv-head) row, written from the same `dtype` (bf16) rows
    kv_format: str = "native"

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def total_lens(self) -> np.ndarray:
        return self.cached_lens + self.new_lens

    # ------------------------------------------------------------------ values
    def _gen(self, stream: int, idx: int) -> torch.Generator:
        g = torch.Generator()
        g.manual_seed(self.seed_values * 1_000_003 + stream * 7919 + idx)
        return g

    def _draw(self, g: torch.Generator, shape) -> torch.Tensor:
        return torch.randn(*shape, generator=g, dtype=torch.float32).to(self.torch_dtype)

    def _owner(self, s: int) -> int:
        """Sequence whose value stream holds the shared prefix of ``s``."""
        if self.pair_of is None or self.pair_of[s] < 0:
            return s
        return min(s, int(self.pair_of[s]))

    def kv_values(self, s: int, start: int, end: int):
        """K and V of sequence ``s`` at logical positions [start, end).

        Shape [end - start, H_kv, D] each, in the storage dtype. Positions
        below the shared prefix come from the pair's common stream, so both
        members of a pair see identical values there. Values are drawn in
        fixed chunks of 4096 positions so any window is reproducible.
        """
        H, D = self.num_kv_heads, self.head_dim
        out_k = torch.empty((max(end - start, 0), H, D), dtype=self.torch_dtype)
        out_v = torch.empty_like(out_k)
        CH = 4096
        pos = start
        while pos < end:
            c = pos // CH
            c0, c1 = c * CH, (c + 1) * CH
            take_end = min(end, c1)
            plen = 0 if self.prefix_len is None else int(self.prefix_len[s])
            if pos < plen:
                take_end = min(take_end, plen)
                src = self._owner(s)
                stream = 1
            else:
                src = s
                stream = 2
            g = self._gen(stream, src * 100_000 + c)
            chunk = self._draw(g, (2, CH, H, D))
            a, b = pos - c0, take_end - c0
            out_k[pos - start: take_end - start] = chunk[0, a:b]
            out_v[pos - start: take_end - start] = chunk[1, a:b]
            pos = take_end
        return out_k, out_v

    def new_kv(self):
        """K/V rows of the tokens written this step, [sum(new_lens), H_kv, D]."""
        ks, vs = [], []
        for s in range(self.num_seqs):
            c, n = int(self.cached_lens[s]), int(self.new_lens[s])
            k, v = self.kv_values(s, c, c + n)
            ks.append(k)
            vs.append(v)
        return torch.cat(ks), torch.cat(vs)

    def queries(self) -> torch.Tensor:
        """Q for this step, [sum(new_lens), H_q, D]."""
        g = self._gen(3, 0)
        n = int(self.new_lens.sum())
        return self._draw(g, (n, self.num_q_heads, self.head_dim))

    def logical_bytes_per_token(self) -> int:
        """Bytes of K plus V one token occupies for one layer (all KV heads);
        FP8 pages: one byte per element plus a 4-byte scale per row."""
        if self.kv_format == "fp8":
            return 2 * self.num_kv_heads * (self.head_dim + 4)
        return 2 * self.num_kv_heads * self.head_dim * self.elem_bytes

    @property
    def pool_torch_dtype(self):
        return torch.float8_e4m3fn if self.kv_format == "fp8" else self.torch_dtype


def _pool_for(rng, blocks_needed: int, factor: float, minimum: int = 0) -> tuple[int, np.ndarray]:
    n = max(int(math.floor(factor * blocks_needed)), minimum, 1)
    return n, rng.permutation(n).astype(np.int32)


def _blocks(n_tokens, block_size):
    return -(-np.asarray(n_tokens, dtype=np.int64) // block_size)


def decode_tiny(scale: float = 1.0) -> Workload:
    rng = np.random.default_rng(1001)
    B = 4
    cached = rng.integers(1, 65, size=B).astype(np.int64)
    n_blk = 128
    return Workload("decode_tiny", "decode", B, 4, 2, 64, 4, "f32", 1.0 / math.sqrt(64),
                    cached, np.ones(B, np.int64), n_blk,
                    rng.permutation(n_blk).astype(np.int32), seed_values=2001)


def decode_gqa(scale: float = 1.0) -> Workload:
    rng = np.random.default_rng(1002)
    B = max(1, int(round(64 * scale)))
    hi = max(128, int(4096 * scale))
    cached = rng.integers(128, hi + 1, size=B).astype(np.int64)
    need = int(_blocks(cached + 1, 16).sum())
    n_blk, order = _pool_for(rng, need, 1.5)
    return Workload("decode_gqa", "decode", B, 32, 8, 128, 16, "bf16", 1.0 / math.sqrt(128),
                    cached, np.ones(B, np.int64), n_blk, order, seed_values=2002)


def decode_mha(scale: float = 1.0) -> Workload:
    rng = np.random.default_rng(1003)
    B = max(1, int(round(256 * scale)))
    hi = max(16, int(2048 * scale))
    cached = np.clip(np.round(rng.lognormal(math.log(512), 1.0, size=B)), 16, hi).astype(np.int64)
    need = int(_blocks(cached + 1, 16).sum())
    n_blk, order = _pool_for(rng, need, 1.5)
    return Workload("decode_mha", "decode", B, 32, 32, 128, 16, "bf16", 1.0 / math.sqrt(128),
                    cached, np.ones(B, np.int64), n_blk, order, seed_values=2003)


def decode_long_shared(scale: float = 1.0, pairs: str = "adjacent") -> Workload:
    """pairs: "adjacent" pairs sequences (0, 1), (2, 3), ...; "far" pairs s
    with s + B/2, so the members of a pair sit half a batch apart."""
    rng = np.random.default_rng(1004)
    B = 8
    lo, hi = max(64, int(32768 * scale)), max(128, int(131072 * scale))
    cached = rng.integers(lo, hi + 1, size=B).astype(np.int64)
    if pairs == "adjacent":
        pair_of = np.array([s ^ 1 for s in range(B)], dtype=np.int64)
    elif pairs == "far":
        pair_of = np.array([(s + B // 2) % B for s in range(B)], dtype=np.int64)
    else:
        raise ValueError("pairs must be 'adjacent' or 'far'")
    prefix = np.zeros(B, np.int64)
    for a in range(B):
        b = int(pair_of[a])
        if a > b:
            continue
        p = int(math.floor(0.75 * min(cached[a], cached[b])))
        if p % 16 == 0:
            p -= 1
        prefix[a] = prefix[b] = p
    # private blocks per member plus the shared ones plus one copy-on-write block per pair
    need = int(_blocks(cached + 1, 16).sum())
    n_blk, order = _pool_for(rng, need, 1.1, minimum=need + 64)
    return Workload("decode_long_shared", "decode", B, 64, 8, 128, 16, "bf16", 1.0 / math.sqrt(128),
                    cached, np.ones(B, np.int64), n_blk, order, pair_of=pair_of,
                    prefix_len=prefix, seed_values=2004)


def prefill(scale: float = 1.0) -> Workload:
    rng = np.random.default_rng(1005)
    B = max(1, int(round(16 * scale)))
    cached = np.full(B, max(16, int(2048 * scale)), np.int64)
    new = np.full(B, max(16, int(512 * scale)), np.int64)
    need = int(_blocks(cached + new, 16).sum())
    n_blk, order = _pool_for(rng, need, 1.5)
    return Workload("prefill", "prefill", B, 32, 8, 128, 16, "bf16", 1.0 / math.sqrt(128),
                    cached, new, n_blk, order, seed_values=2005)


def with_fp8_pages(wl: Workload) -> Workload:
    """The same workload (structure and bf16 values) stored in FP8 pages."""
    if wl.dtype != "bf16":
        raise ValueError("FP8 pages are written from bf16 rows")
    return dataclasses.replace(wl, name=wl.name + "_fp8", kv_format="fp8")


def decode_gqa_fp8(scale: float = 1.0) -> Workload:
    """The GQA decode batch with FP8 (E4M3) pages."""
    return with_fp8_pages(decode_gqa(scale))


def decode_long_shared_fp8(scale: float = 1.0) -> Workload:
    """The long shared-prefix decode batch with FP8 (E4M3) pages."""
    return with_fp8_pages(decode_long_shared(scale))


WORKLOADS = {
    "decode_tiny": decode_tiny,
    "decode_gqa": decode_gqa,
    "decode_gqa_fp8": decode_gqa_fp8,
    "decode_long_shared_fp8": decode_long_shared_fp8,
    "decode_mha": decode_mha,
    "decode_long_shared": decode_long_shared,
    "prefill": prefill,
}


def custom_decode(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, dtype,
                  cached_lens, seed=7, pool_factor=1.5, new_lens=None, kind="decode",
                  causal=True) -> Workload:
    """A small hand-shaped workload for edge-case tests."""
    rng = np.random.default_rng(seed)
    cached = np.asarray(cached_lens, dtype=np.int64)
    new = np.ones(num_seqs, np.int64) if new_lens is None else np.asarray(new_lens, np.int64)
    need = int(_blocks(cached + new, block_size).sum())
    n_blk, order = _pool_for(rng, need, pool_factor, minimum=need + 2)
    return Workload("custom", kind, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                    dtype, 1.0 / math.sqrt(head_dim), cached, new, n_blk, order,
                    causal=causal, seed_values=seed + 5000)

"""Host-side block manager used to lay out synthetic workloads.

This is the bookkeeping half of PagedAttention, as the pages describe it:

* a pool of identical physical blocks handed out from a free list, with a
  reference count per block ("PagedAttention: paging the KV cache", pofe.ai,
  §How it works and §Sharing and copy-on-write; "PagedAttention: Virtual-Memory
  KV Cache Management, Continuous Batching, and PyTorch Architecture",
  ailinkdeeptech.com, §4 Automatic Prefix Caching and Copy-on-Write);
* one block table per sequence: entry j is the physical id of logical block j;
* allocation on demand: a new block only when the last one is full;
* fork (every block shared, refcount + 1) and copy-on-write when a sequence
  appends into a shared, partially filled last block.

It decides *which* physical block holds which logical block and records the
(src, dst) pairs a copy-on-write needs. It does no slot arithmetic and no
attention arithmetic: those belong to the kernels and to the oracle, which both
take the tables produced here as inputs.
"""
from __future__ import annotations

from collections import deque
from typing import Iterable, List, Optional, Tuple


class PoolExhausted(MemoryError):
    """Raised when an allocation finds the free list empty (the point where a
    serving engine would preempt a sequence)."""


class BlockPool:
    """Free list + reference counts over ``num_blocks`` physical blocks."""

    def __init__(self, num_blocks: int, block_size: int,
                 free_order: Optional[Iterable[int]] = None) -> None:
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        order = list(range(num_blocks)) if free_order is None else [int(i) for i in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of range(num_blocks)")
        self.free: deque[int] = deque(order)
        self.ref: List[int] = [0] * num_blocks

    @property
    def num_free(self) -> int:
        return len(self.free)

    def alloc(self) -> int:
        if not self.free:
            raise PoolExhausted("no free block: a sequence must be preempted")
        i = self.free.popleft()
        self.ref[i] = 1
        return i

    def take(self, i: int) -> int:
        """Allocate a specific free block (used to pin a table to given ids)."""
        self.free.remove(i)
        self.ref[i] = 1
        return i

    def share(self, i: int) -> int:
        if self.ref[i] <= 0:
            raise ValueError(f"block {i} is not live")
        self.ref[i] += 1
        return i

    def release(self, i: int) -> None:
        if self.ref[i] <= 0:
            raise ValueError(f"block {i} released more often than referenced")
        self.ref[i] -= 1
        if self.ref[i] == 0:
            self.free.append(i)


class SeqTable:
    """One sequence's block table and length."""

    def __init__(self, pool: BlockPool) -> None:
        self.pool = pool
        self.table: List[int] = []
        self.length = 0

    def blocks_needed(self, n_tokens: int) -> int:
        b = self.pool.block_size
        return -(-n_tokens // b)

    def admit(self, prompt_len: int) -> None:
        """Allocate the blocks a prompt of ``prompt_len`` tokens fills (prefill)."""
        if self.table or self.length:
            raise ValueError("admit() on a non-empty sequence")
        need = self.blocks_needed(prompt_len)
        if need > self.pool.num_free:
            raise PoolExhausted("prompt does not fit in the free pool")
        self.table = [self.pool.alloc() for _ in range(need)]
        self.length = prompt_len

    def fork(self) -> "SeqTable":
        """A new sequence sharing every block of this one (parallel sampling)."""
        child = SeqTable(self.pool)
        child.table = [self.pool.share(i) for i in self.table]
        child.length = self.length
        return child

    def append(self) -> Optional[Tuple[int, int]]:
        """Make room for one more token; return a (src, dst) copy-on-write pair or None.

        A fresh block is taken when the last one is full; when the last block is
        partially filled and shared, it is copied to a fresh block first and the
        table is remapped, so the write that follows touches a private block.
        """
        b = self.pool.block_size
        pair = None
        if self.length % b == 0:
            self.table.append(self.pool.alloc())
        elif self.pool.ref[self.table[-1]] > 1:
            old = self.table[-1]
            new = self.pool.alloc()
            self.pool.release(old)
            self.table[-1] = new
            pair = (old, new)
        self.length += 1
        return pair

    def free(self) -> None:
        for i in self.table:
            self.pool.release(i)
        self.table = []
        self.length = 0


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int,
                       dtype_bytes: int) -> int:
    """Cache bytes one token occupies: 2 (K and V) x layers x KV heads x head_dim x sizeof.

    The memory formula M_KV of "PagedAttention: Virtual-Memory KV Cache
    Management, ..." §KV Cache Memory Bottlenecks, per token.
    """
    return 2 * num_layers * num_kv_heads * head_dim * dtype_bytes

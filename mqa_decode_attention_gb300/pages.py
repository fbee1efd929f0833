"""Host-side page allocator: block tables for the paged cache.

Follows the allocation policy of the pages' PagedKVCache ("KV Cache 최적화
심층 분석", youngju.dev): a FIFO free list of physical blocks, a new block
taken when a sequence's length reaches a block boundary, an out-of-memory
error when the free list is empty, and blocks returned on free. The device
kernels only read the table; this class only writes it (host memory), and
``table()`` packs it into the int32 [batch, max_pages] layout the C ABI takes,
unused entries -1.
"""

from __future__ import annotations

from collections import deque

import torch


class PagePool:
    def __init__(self, num_pages: int, page_size: int = 16):
        if num_pages < 1 or page_size < 1:
            raise ValueError("num_pages and page_size must be positive")
        self.page_size = page_size
        self.num_pages = num_pages
        self.free = deque(range(num_pages))
        self.blocks: dict[int, list[int]] = {}
        self.lengths: dict[int, int] = {}

    def _take(self) -> int:
        if not self.free:
            raise RuntimeError("out of KV pages: no free block left in the pool")
        return self.free.popleft()

    def add_sequence(self, seq: int) -> None:
        if seq in self.blocks:
            raise ValueError(f"sequence {seq} already allocated")
        self.blocks[seq] = []
        self.lengths[seq] = 0

    def reserve(self, seq: int, n_tokens: int = 1) -> int:
        """Grow sequence ``seq`` by n_tokens, taking pages at block boundaries.
        Returns the position of the last new token (the append position)."""
        for _ in range(n_tokens):
            L = self.lengths[seq]
            if L % self.page_size == 0:
                self.blocks[seq].append(self._take())
            self.lengths[seq] = L + 1
        return self.lengths[seq] - 1

    def slot(self, seq: int, pos: int) -> tuple[int, int]:
        """(physical page, row) of token ``pos`` of sequence ``seq``."""
        return self.blocks[seq][pos // self.page_size], pos % self.page_size

    def release(self, seq: int) -> None:
        for b in self.blocks.pop(seq):
            self.free.append(b)
        del self.lengths[seq]

    def table(self, seqs: list[int], max_pages: int | None = None) -> torch.Tensor:
        mp = max_pages or max(1, max(len(self.blocks[s]) for s in seqs))
        t = torch.full((len(seqs), mp), -1, dtype=torch.int32)
        for i, s in enumerate(seqs):
            row = self.blocks[s]
            if len(row) > mp:
                raise ValueError(f"sequence {s} holds {len(row)} pages, table has {mp}")
            t[i, :len(row)] = torch.tensor(row, dtype=torch.int32)
        return t

    def seq_lens(self, seqs: list[int]) -> torch.Tensor:
        return torch.tensor([self.lengths[s] for s in seqs], dtype=torch.int32)

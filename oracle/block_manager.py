"""Plain reference of a paged KV-cache block manager (test infrastructure only).

Only the tests may import this module; the product library never calls it.

What it models ("Inference optimization" lesson, section "PagedAttention";
"Continuous Batching e PagedAttention no vLLM", section 3):

  * The cache is a pool of fixed-size pages (16 tokens each) that may sit
    anywhere in memory.  Each request owns a page table mapping its logical
    blocks (token t lives in logical block t // 16 at offset t % 16) to
    physical pages.  A request grows by one page when its last page is full;
    the last page may be partly filled.
  * Pages of a shared prefix (a system prompt used by many requests) are
    stored once and referenced by every request that shares it.  A request
    gets its own page only when it diverges: writing a token into a page that
    others still reference first copies that page (copy-on-write).
  * A finished request returns its pages; a page goes back to the pool when
    no request references it any more.

Readings where the pages are silent: a free page is taken lowest id first
(any free page is valid; a fixed choice makes tables reproducible); a fork
shares every page of the parent, including its partly filled last page; only
that last page can need a copy, because appends never touch earlier pages.
Slots follow slot = page_id * 16 + offset.
"""
from __future__ import annotations

import heapq


class BlockManagerError(Exception):
    pass


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int = 16, max_blocks_per_seq: int = 1 << 30):
        if num_blocks <= 0 or block_size <= 0 or max_blocks_per_seq <= 0:
            raise BlockManagerError("invalid sizes")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.max_blocks_per_seq = max_blocks_per_seq
        self.free = list(range(num_blocks))  # a heap: lowest id first
        heapq.heapify(self.free)
        self.ref = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}

    # ------------------------------------------------------------ pool
    def num_free(self) -> int:
        return len(self.free)

    def _take(self) -> int:
        if not self.free:
            raise BlockManagerError("out of blocks")
        b = heapq.heappop(self.free)
        assert self.ref[b] == 0
        self.ref[b] = 1
        return b

    def _drop(self, b: int) -> None:
        self.ref[b] -= 1
        assert self.ref[b] >= 0
        if self.ref[b] == 0:
            heapq.heappush(self.free, b)

    def _slot(self, seq: int, t: int) -> int:
        return self.tables[seq][t // self.block_size] * self.block_size + t % self.block_size

    # -------------------------------------------------------- requests
    def add(self, seq: int, num_tokens: int) -> list[int]:
        """A new request with a prompt of num_tokens; returns the prompt's slots."""
        if seq in self.tables or num_tokens < 0:
            raise BlockManagerError("bad add")
        need = -(-num_tokens // self.block_size)
        if need > self.max_blocks_per_seq:
            raise BlockManagerError("sequence too long")
        if need > len(self.free):
            raise BlockManagerError("out of blocks")
        self.tables[seq] = [self._take() for _ in range(need)]
        self.lens[seq] = num_tokens
        return [self._slot(seq, t) for t in range(num_tokens)]

    def fork(self, parent: int, child: int) -> None:
        """child starts as a copy of parent that shares all of its pages."""
        if parent not in self.tables or child in self.tables:
            raise BlockManagerError("bad fork")
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            self.ref[b] += 1

    def append(self, seq: int) -> tuple[int, list[tuple[int, int]]]:
        """Reserve the slot of the next token of seq.

        Returns (slot, copies): copies lists (src, dst) page pairs whose
        contents must be copied before the token is written.
        """
        if seq not in self.tables:
            raise BlockManagerError("unknown sequence")
        t = self.lens[seq]
        table = self.tables[seq]
        copies = []
        if t % self.block_size == 0:          # last page full (or none yet): a new page
            if len(table) + 1 > self.max_blocks_per_seq:
                raise BlockManagerError("sequence too long")
            table.append(self._take())
        else:
            last = table[-1]
            if self.ref[last] > 1:            # shared and about to be written: copy it
                new = self._take()
                copies.append((last, new))
                self._drop(last)
                table[-1] = new
        self.lens[seq] = t + 1
        return self._slot(seq, t), copies

    def free_seq(self, seq: int) -> None:
        if seq not in self.tables:
            raise BlockManagerError("unknown sequence")
        for b in self.tables.pop(seq):
            self._drop(b)
        del self.lens[seq]

    def table(self, seq: int) -> list[int]:
        return list(self.tables[seq])

    def length(self, seq: int) -> int:
        return self.lens[seq]

"""Paged KV bookkeeping: capacity reservation and rewind with LIFO page release.
TEST INFRASTRUCTURE.

  [TS] "the shared loop": SpecEnsureCapacity(requiredSeqLen) and
       SpecRewindCache(length) on the trunk; CacheSeqLen.
  [PI] "the transaction", Commit / roll back: accepted tokens' KV is committed
       and the unused tail of the speculative reservation is LIFO-dropped.
  [PI] "context limit": a request that does not fit is rejected cleanly at
       admission rather than crashing.
  [CA] "dense rollback": rollback is "do not advance"; rows past the new
       length are stale, never read, and overwritten by the next forward.

Readings where the pages are silent:
  * the free pool is a stack; the first pop returns page 0, then 1, ...;
  * ensure_capacity serves sequences b = 0..B-1 in order, each taking pages
    for its page-table slots in ascending order; it is all-or-nothing: if any
    sequence would exceed its page-table size or the pool runs dry, nothing
    changes and the call fails;
  * rewind releases, for b = B-1 down to 0, each sequence's pages past
    ceil(length / page_size), highest slot first. A rewind to the lengths held
    before an ensure_capacity therefore restores the pool exactly: the pages
    go back in the reverse of the order they were taken.
"""
from __future__ import annotations


class CapacityError(Exception):
    pass


def pages_for(length: int, page_size: int) -> int:
    return -(-length // page_size)


class PagePool:
    def __init__(self, n_pages: int, page_size: int, max_batch: int, max_pages_per_seq: int):
        self.page_size = page_size
        self.max_pages_per_seq = max_pages_per_seq
        self.free = list(range(n_pages - 1, -1, -1))     # top of the stack is the end of the list
        self.table = [[] for _ in range(max_batch)]
        self.length = [0] * max_batch                     # written length per sequence

    def ensure_capacity(self, required: list) -> None:
        """Give sequence b enough pages for required[b] tokens (a negative entry skips b)."""
        need = []
        for b, r in enumerate(required):
            n = pages_for(r, self.page_size) if r >= 0 else 0
            if n > self.max_pages_per_seq:
                raise CapacityError(f"sequence {b}: {r} tokens exceed the page table")
            need.append(max(0, n - len(self.table[b])))
        if sum(need) > len(self.free):
            raise CapacityError("out of pages")
        for b, n in enumerate(need):
            for _ in range(n):
                self.table[b].append(self.free.pop())

    def set_length(self, b: int, length: int) -> None:
        self.length[b] = length

    def rewind(self, lengths: list) -> None:
        """Set each cache length (a negative entry skips b) and release pages past it, LIFO."""
        for b, r in enumerate(lengths):
            if r >= 0 and r > self.length[b]:
                raise ValueError(f"sequence {b}: rewind to {r} past the written length {self.length[b]}")
        for b in range(len(lengths) - 1, -1, -1):
            r = lengths[b]
            if r < 0:
                continue
            keep = pages_for(r, self.page_size)
            while len(self.table[b]) > keep:
                self.free.append(self.table[b].pop())
            self.length[b] = r

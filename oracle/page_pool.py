"""Block pool and per-request block table, restated -- TEST INFRASTRUCTURE ONLY.

Source: "Aufmerksamkeit" feed (chatgpz.de), PagedAttention article,
SECTION 2 "Pages + Block Table" (classes PagePool and PagedRequest) and
SECTION 3 "Copy-on-Write: Shared System Prompts".

The pool keeps a FIFO free list (allocation takes the head, release appends
to the tail) and a reference count per live page:
  allocate   -> head of the free list, refcount 1; an empty list is an OOM
  release    -> refcount - 1; at zero the page returns to the tail of the list
  share      -> refcount + 1, no new page
  cow_copy   -> allocate a fresh page, then release the old one
  utilisation-> (total - free) / total * 100
A request appends tokens one at a time and claims a new page whenever its
token count is a multiple of the page size.

Readings where the article is silent (the article's dict would silently
misbehave): releasing or sharing a page that is not live, and an id outside
the pool, raise ``ValueError``.
"""
from __future__ import annotations

from collections import deque


class PoolOOM(MemoryError):
    pass


class PagePool:
    def __init__(self, total_pages: int):
        self.total = int(total_pages)
        self.free = deque(range(self.total))
        self.ref_count: dict[int, int] = {}

    def _live(self, pid: int):
        if not (0 <= pid < self.total) or pid not in self.ref_count:
            raise ValueError(f"page {pid} is not live")

    def allocate(self) -> int:
        if not self.free:
            raise PoolOOM("no free pages")
        pid = self.free.popleft()
        self.ref_count[pid] = 1
        return pid

    def release(self, pid: int) -> None:
        self._live(pid)
        self.ref_count[pid] -= 1
        if self.ref_count[pid] <= 0:
            del self.ref_count[pid]
            self.free.append(pid)

    def share(self, pid: int) -> None:
        self._live(pid)
        self.ref_count[pid] += 1

    def cow_copy(self, pid: int) -> int:
        self._live(pid)
        new_pid = self.allocate()
        self.release(pid)
        return new_pid

    def refcount(self, pid: int) -> int:
        return self.ref_count.get(pid, 0)

    @property
    def utilisation(self) -> float:
        return (self.total - len(self.free)) / self.total * 100.0


class PagedRequest:
    def __init__(self, req_id, pool: PagePool, page_size: int = 16):
        self.id = req_id
        self.pool = pool
        self.page_size = page_size
        self.block_table: list[int] = []
        self.tokens = 0

    def generate_token(self) -> None:
        if self.tokens % self.page_size == 0:
            self.block_table.append(self.pool.allocate())
        self.tokens += 1

    def free(self) -> None:
        for pid in self.block_table:
            self.pool.release(pid)
        self.block_table.clear()

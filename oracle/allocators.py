"""Plain restatement of GraniKV's two KV pools.  TEST INFRASTRUCTURE ONLY.

Only the tests, the package's smoke check and the benchmark's CPU-baseline leg may import
this module.

HOT pool ("3 GraniKV", asymmetric KV-cache paging; "B.8 Multi-prefix sensitivity", mixed slab
sizes exercise first-fit packing; "B.10 Cross-pool admission and promotion policy"): one
contiguous slab per prefix.  Allocation takes the lowest-offset free extent that can hold
L_p slots and carves the slab from its start; a request that no extent can hold fails (the
caller then places the prefix in COLD); nothing is ever moved or demoted.  The card page calls
the allocator a bump pointer: with no frees, lowest-offset first fit is exactly a bump
pointer.  Freeing returns the extent and merges it with free neighbours.  Slab ids are the
lowest unused id.

COLD pool ("1 Introduction" and "3 GraniKV": page size 1 for suffix and decoded tokens; the
card page: a token-level free list): a FIFO ring of free slot ids.  An allocation of n_new[b]
tokens for each request b gives request b the ring entries starting at
head + (exclusive prefix sum of n_new)[b], in request order, appends them to the request's
token table and bumps its length.  It is all-or-nothing: if fewer free slots remain than the
total asked, nothing is popped.  Freeing appends slot ids at the tail in the given order.

Parity of this module is pinned by hand-derived scripted scenarios in tests/golden/.
"""

from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple


class NoHotSpace(Exception):
    pass


class NoColdSpace(Exception):
    pass


class HotFirstFit:
    """First-fit allocator over HOT slots [0, n_hot)."""

    def __init__(self, n_hot: int, max_slabs: int = 1 << 30):
        self.n_hot = int(n_hot)
        self.max_slabs = int(max_slabs)
        self.free: List[List[int]] = [[0, self.n_hot]] if self.n_hot > 0 else []  # [off, len]
        self.slabs: Dict[int, Tuple[int, int]] = {}

    def alloc(self, L_p: int) -> Tuple[int, int]:
        if L_p <= 0:
            raise ValueError("L_p must be positive")
        sid = 0
        while sid in self.slabs:
            sid += 1
        if sid >= self.max_slabs:
            raise NoHotSpace("slab table full")
        for ext in self.free:  # kept sorted by offset
            if ext[1] >= L_p:
                off = ext[0]
                ext[0] += L_p
                ext[1] -= L_p
                if ext[1] == 0:
                    self.free.remove(ext)
                self.slabs[sid] = (off, L_p)
                return sid, off
        raise NoHotSpace(f"no free extent of {L_p} slots")

    def free_slab(self, sid: int) -> None:
        off, ln = self.slabs.pop(sid)
        self.free.append([off, ln])
        self.free.sort()
        merged: List[List[int]] = []
        for e in self.free:
            if merged and merged[-1][0] + merged[-1][1] == e[0]:
                merged[-1][1] += e[1]
            else:
                merged.append(list(e))
        self.free = merged

    def largest_free(self) -> int:
        return max((e[1] for e in self.free), default=0)


class ColdRing:
    """FIFO ring of free COLD slot ids with per-request token tables."""

    def __init__(self, initial: Sequence[int]):
        self.ring: List[int] = [int(x) for x in initial]
        self.capacity = len(self.ring)
        self.head = 0            # entries [head, tail) are free
        self.tail = len(self.ring)

    @property
    def n_free(self) -> int:
        return self.tail - self.head

    def _at(self, pos: int) -> int:
        return self.ring[pos % self.capacity]

    def alloc(self, n_new: Sequence[int], tables: List[List[int]], cap: Optional[int] = None
              ) -> List[int]:
        """Pop sum(n_new) slots; request b gets the next n_new[b] in request order.

        Appends to ``tables[b]`` and returns the popped slots in order.
        """
        total = sum(int(x) for x in n_new)
        if total > self.n_free:
            raise NoColdSpace(f"asked {total}, {self.n_free} free")
        if cap is not None:
            for b, n in enumerate(n_new):
                if len(tables[b]) + int(n) > cap:
                    raise ValueError(f"request {b} exceeds table capacity {cap}")
        out: List[int] = []
        pos = self.head
        for b, n in enumerate(n_new):
            for _ in range(int(n)):
                slot = self._at(pos)
                tables[b].append(slot)
                out.append(slot)
                pos += 1
        self.head = pos
        return out

    def free(self, slots: Sequence[int]) -> None:
        if len(slots) > self.capacity - self.n_free:
            raise ValueError("freeing more slots than are allocated")
        for s in slots:
            self.ring[self.tail % self.capacity] = int(s)
            self.tail += 1

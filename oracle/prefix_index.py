"""Plain restatement of GraniKV's prefix lifecycle.  TEST INFRASTRUCTURE ONLY.

Only the tests, the package's smoke check and the benchmark's CPU-baseline leg may import
this module.

What it restates (GraniKV, arXiv:2608.15584):
  * "2 Related Work", prefix-aware serving: cached prefixes are indexed by their token-id
    sequences for longest-prefix reuse, and a cached prefix is kept while a reference count
    says active requests depend on it;
  * card page: one HOT slab per prefix node, one index for both pools;
  * "B.10 Cross-pool admission and promotion policy": a new prefix goes to HOT first and needs
    L_p contiguous slots there; when HOT has no such extent it is placed in COLD; prefixes in
    HOT are never demoted.

Readings where the pages leave a step open (the library's index follows the same ones):
  * a request reuses the longest admitted prefix that its token sequence starts with, whole;
  * only unreferenced prefixes may be evicted, least recently used first, and an admission
    evicts HOT prefixes only if evicting every unreferenced HOT prefix would make the new one
    fit (then as few as LRU order needs); otherwise it evicts nothing and places it in COLD;
  * the use clock advances on insert (also of an already-admitted sequence), on a match that
    takes a reference, on acquire and on release;
  * prefix handles count up from 0 and are never reused.

No tree here: the admitted prefixes are a dict keyed by their token tuples, and a match is a
scan over all of them.  Parity of this module is pinned by the hand-derived scenario
tests/golden/prefix_lifecycle_scenario.txt.
"""

from __future__ import annotations

import copy
from typing import Dict, List, Optional, Sequence, Tuple

from .allocators import HotFirstFit, NoHotSpace


class PrefixIndexOracle:
    def __init__(self, n_hot: int, max_slabs: int = 1024):
        self.hot = HotFirstFit(n_hot, max_slabs=max_slabs)
        self.entries: Dict[int, dict] = {}   # handle -> {tokens, slab, offset, refs, used}
        self.next_id = 0
        self.clock = 0

    def _tick(self) -> int:
        self.clock += 1
        return self.clock

    def info(self, pid: int) -> dict:
        e = self.entries[pid]
        return {"prefix_id": pid, "length": len(e["tokens"]), "slab_id": e["slab"],
                "refcount": e["refs"], "slot_offset": e["offset"]}

    @staticmethod
    def _none() -> dict:
        return {"prefix_id": -1, "length": 0, "slab_id": -1, "refcount": 0, "slot_offset": -1}

    def match(self, tokens: Sequence[int], acquire: bool = False) -> dict:
        t = tuple(int(x) for x in tokens)
        best: Optional[int] = None
        for pid, e in self.entries.items():
            p = e["tokens"]
            if len(p) <= len(t) and t[:len(p)] == p:
                if best is None or len(p) > len(self.entries[best]["tokens"]):
                    best = pid
        if best is None:
            return self._none()
        if acquire:
            self.entries[best]["refs"] += 1
            self.entries[best]["used"] = self._tick()
        return self.info(best)

    def _fits(self, hot: HotFirstFit, n: int) -> bool:
        return hot.largest_free() >= n and len(hot.slabs) < hot.max_slabs

    def insert(self, tokens: Sequence[int]) -> Tuple[dict, List[int]]:
        t = tuple(int(x) for x in tokens)
        if not t:
            raise ValueError("empty prefix")
        for pid, e in self.entries.items():
            if e["tokens"] == t:
                e["used"] = self._tick()
                return self.info(pid), []
        n = len(t)
        victims: List[int] = []
        hot_ok = self._fits(self.hot, n)
        if not hot_ok:
            idle = sorted((e["used"], pid) for pid, e in self.entries.items()
                          if e["refs"] == 0 and e["slab"] >= 0)
            trial = copy.deepcopy(self.hot)
            for _, pid in idle:
                trial.free_slab(self.entries[pid]["slab"])
                victims.append(pid)
                if self._fits(trial, n):
                    hot_ok = True
                    break
            if not hot_ok:
                victims = []
        for pid in victims:
            self.hot.free_slab(self.entries.pop(pid)["slab"])
        slab, offset = -1, -1
        if hot_ok:
            slab, offset = self.hot.alloc(n)
        pid = self.next_id
        self.next_id += 1
        self.entries[pid] = {"tokens": t, "slab": slab, "offset": offset, "refs": 0,
                             "used": self._tick()}
        return self.info(pid), victims

    def acquire(self, pid: int) -> None:
        e = self.entries[pid]  # KeyError for an unknown handle
        e["refs"] += 1
        e["used"] = self._tick()

    def release(self, pid: int) -> None:
        e = self.entries[pid]
        if e["refs"] <= 0:
            raise ValueError("release of an unreferenced prefix")
        e["refs"] -= 1
        e["used"] = self._tick()

    def remove(self, pid: int) -> None:
        e = self.entries[pid]
        if e["refs"] != 0:
            raise ValueError("remove of a referenced prefix")
        if e["slab"] >= 0:
            self.hot.free_slab(e["slab"])
        del self.entries[pid]

    def n_nodes(self) -> int:
        """Nodes of the smallest path-compressed tree holding the admitted sequences: every
        non-empty token string that is an admitted prefix, or that two admitted prefixes
        continue with different next tokens."""
        seqs = {e["tokens"] for e in self.entries.values()}
        nxt: Dict[tuple, set] = {}  # every non-empty prefix string -> tokens that follow it
        for s in seqs:
            for i in range(1, len(s) + 1):
                nxt.setdefault(s[:i], set())
                if i < len(s):
                    nxt[s[:i]].add(s[i])
        return sum(1 for p, follow in nxt.items() if p in seqs or len(follow) >= 2)

    def stats(self) -> Tuple[int, int, int]:
        n_hot = sum(1 for e in self.entries.values() if e["slab"] >= 0)
        return len(self.entries), n_hot, self.n_nodes()


__all__ = ["PrefixIndexOracle", "NoHotSpace"]

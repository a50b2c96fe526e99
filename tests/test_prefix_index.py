"""Prefix lifecycle (no GPU): the oracle's restatement against the hand-derived scenario, and
libgranikv's radix-tree index against the oracle, on the scenario and on seeded random
operation sequences.

GraniKV (arXiv:2608.15584): "2 Related Work" (prefix-aware serving, reference-counted radix
index over token ids), the card page (one HOT slab per prefix node) and "B.10 Cross-pool
admission and promotion policy" (HOT first, COLD fallback, no demotion)."""

import os

import numpy as np
import pytest

from oracle.prefix_index import PrefixIndexOracle
from shared_prefix_kv_decode_gb300 import _binding as gb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SCENARIO = os.path.join(ROOT, "tests", "golden", "prefix_lifecycle_scenario.txt")


class Invalid(Exception):
    pass


class OracleSide:
    def __init__(self, n_hot, max_slabs):
        self.x = PrefixIndexOracle(n_hot, max_slabs=max_slabs)

    def _call(self, fn, *a):
        try:
            return fn(*a)
        except (KeyError, ValueError) as e:
            raise Invalid(str(e))

    def insert(self, seq):
        return self.x.insert(seq)

    def match(self, seq, acquire):
        return self.x.match(seq, acquire)

    def acquire(self, pid):
        self._call(self.x.acquire, pid)

    def release(self, pid):
        self._call(self.x.release, pid)

    def remove(self, pid):
        self._call(self.x.remove, pid)

    def stats(self):
        return self.x.stats()


class LibrarySide:
    def __init__(self, n_hot, max_slabs):
        # host-only context whose HOT pool is n_hot slots (n_hot = n_slots / 2)
        self.ctx = gb.Context(n_layers=1, n_q=32, n_kv=8, head_dim=128, dtype=gb.DTYPE_BF16,
                              n_slots=2 * n_hot, hot_fraction=0.5, max_slabs=max_slabs, host_only=True)
        assert self.ctx.hot_stats()[0] == n_hot
        self.x = self.ctx.index()

    def _call(self, fn, *a):
        try:
            return fn(*a)
        except gb.GranikvError as e:
            if e.status != gb.ERR_INVALID:
                raise
            raise Invalid(str(e))

    def insert(self, seq):
        return self.x.insert(seq)

    def match(self, seq, acquire):
        return self.x.match(seq, acquire)

    def acquire(self, pid):
        self._call(self.x.acquire, pid)

    def release(self, pid):
        self._call(self.x.release, pid)

    def remove(self, pid):
        self._call(self.x.remove, pid)

    def stats(self):
        return self.x.stats()


def _seq(text):
    out = []
    for run in text.split(","):
        tok, cnt = run.split(":")
        out += [int(tok)] * int(cnt)
    return out


def run_scenario(make_side):
    side = None
    n_checked = 0
    with open(SCENARIO) as f:
        for raw in f:
            line = raw.split("#")[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "pool":
                side = make_side(int(tok[1]), int(tok[2]))
                continue
            op = tok[0]
            if op == "insert":
                info, evicted = side.insert(_seq(tok[1]))
                want = tok[3:tok.index("|")]
                got = [str(info["prefix_id"])]
                if info["slab_id"] >= 0:
                    got += ["HOT", str(info["slab_id"]), str(info["slot_offset"])]
                else:
                    got += ["COLD"]
                    assert info["slot_offset"] == -1, line
                assert got == want, line
                want_ev = tok[tok.index("evicted") + 1:]
                assert [str(e) for e in evicted] == ([] if want_ev == ["-"] else want_ev), line
            elif op == "match":
                acquire = "acquire" in tok
                info = side.match(_seq(tok[1]), acquire)
                want = tok[tok.index("->") + 1:]
                if want == ["none"]:
                    assert info["prefix_id"] == -1, line
                else:
                    assert [info["prefix_id"], info["length"], info["refcount"]] == [int(w) for w in want], line
            elif op in ("acquire", "release", "remove"):
                fn = getattr(side, op)
                if tok[-1] == "INVALID":
                    with pytest.raises(Invalid):
                        fn(int(tok[1]))
                else:
                    fn(int(tok[1]))
            elif op == "stats":
                assert list(side.stats()) == [int(w) for w in tok[2:]], line
            else:
                raise ValueError(line)
            n_checked += 1
    return n_checked


def test_oracle_on_hand_derived_scenario():
    assert run_scenario(OracleSide) == 44


def test_library_index_on_hand_derived_scenario(granikv_lib):
    assert run_scenario(LibrarySide) == 44


def _random_seq(rng, stems):
    """A token sequence that often shares a stem with earlier ones, so that the tree splits,
    nests and folds."""
    if stems and rng.random() < 0.7:
        base = list(stems[int(rng.integers(len(stems)))])
        cut = int(rng.integers(1, len(base) + 1))
        seq = base[:cut]
    else:
        seq = []
    for _ in range(int(rng.integers(0 if seq else 1, 3))):
        seq += [int(rng.integers(0, 3))] * int(rng.integers(1, 25))
    return seq


@pytest.mark.parametrize("seed", range(6))
def test_library_index_matches_oracle_on_random_operations(granikv_lib, seed):
    rng = np.random.default_rng(seed)
    n_hot = int(rng.integers(60, 160))
    max_slabs = int(rng.integers(3, 9))
    lib, ora = LibrarySide(n_hot, max_slabs), OracleSide(n_hot, max_slabs)
    stems = []
    handles = []
    held_slab = {}  # handle -> slab offset while it is referenced (no-demotion check)
    for step in range(800):
        r = rng.random()
        if r < 0.35:
            seq = _random_seq(rng, stems)
            stems.append(seq)
            a, b = lib.insert(seq), ora.insert(seq)
            assert a == b, (step, seq)
            handles.append(a[0]["prefix_id"])
            for ev in a[1]:
                assert ev not in held_slab, "a referenced prefix was evicted"
        elif r < 0.6:
            seq = _random_seq(rng, stems)
            acq = bool(rng.random() < 0.6)
            a, b = lib.match(seq, acq), ora.match(seq, acq)
            assert a == b, (step, seq)
            if acq and a["prefix_id"] >= 0:
                held_slab[a["prefix_id"]] = (a["slab_id"], a["slot_offset"])
        else:
            op = ("release", "acquire", "remove")[int(rng.integers(3))]
            pid = int(rng.choice(handles)) if handles and rng.random() < 0.9 else int(rng.integers(0, 50))
            outcomes = []
            for side in (lib, ora):
                try:
                    getattr(side, op)(pid)
                    outcomes.append("ok")
                except Invalid:
                    outcomes.append("invalid")
            assert outcomes[0] == outcomes[1], (step, op, pid)
            if outcomes[0] == "ok" and op == "acquire":
                info = lib.x.info(pid)
                held_slab[pid] = (info["slab_id"], info["slot_offset"])
        if step % 20 == 0 or step == 799:
            assert lib.stats() == ora.stats(), step
        # referenced prefixes stay where they are; live HOT slabs are disjoint and in range
        live = {pid: ora.x.info(pid) for pid in ora.x.entries}
        for pid in list(held_slab):
            if pid not in live or live[pid]["refcount"] == 0:
                del held_slab[pid]
                continue
            assert (live[pid]["slab_id"], live[pid]["slot_offset"]) == held_slab[pid], "demoted or moved"
        spans = sorted((i["slot_offset"], i["length"]) for i in live.values() if i["slab_id"] >= 0)
        for (o1, l1), (o2, _) in zip(spans, spans[1:]):
            assert o1 + l1 <= o2
        assert all(0 <= o and o + l <= n_hot for o, l in spans)
    assert len(handles) > 150


def test_index_argument_errors(granikv_lib):
    lib = LibrarySide(100, 4)
    with pytest.raises(gb.GranikvError):
        lib.x.insert([])
    assert lib.x.match([])["prefix_id"] == -1
    with pytest.raises(gb.GranikvError):
        lib.x.info(0)


def test_index_destroy_returns_its_slabs(granikv_lib):
    side = LibrarySide(100, 4)
    side.x.insert([1] * 60)
    side.x.insert([2] * 30)
    assert side.ctx.hot_stats() == (100, 10)
    side.x.close()
    assert side.ctx.hot_stats() == (100, 100)


# planted mistakes in the oracle: each must be caught by the hand-derived scenario

class _ShortestMatch(PrefixIndexOracle):
    def match(self, tokens, acquire=False):
        t = tuple(int(x) for x in tokens)
        hits = [pid for pid, e in self.entries.items() if t[:len(e["tokens"])] == e["tokens"]]
        if not hits:
            return self._none()
        best = min(hits, key=lambda pid: len(self.entries[pid]["tokens"]))
        if acquire:
            self.acquire(best)
        return self.info(best)


class _MostRecentlyUsedEviction(PrefixIndexOracle):
    def _tick(self):
        self.clock -= 1  # later use sorts first: evicts the most recently used
        return self.clock


class _FutileEviction(PrefixIndexOracle):
    def insert(self, tokens):
        # evicts every idle HOT prefix whenever the new one does not fit at once
        t = tuple(int(x) for x in tokens)
        if not any(e["tokens"] == t for e in self.entries.values()) and not self._fits(self.hot, len(t)):
            for pid in [p for p, e in self.entries.items() if e["refs"] == 0 and e["slab"] >= 0]:
                self.hot.free_slab(self.entries.pop(pid)["slab"])
        return super().insert(tokens)


class _HandlesReused(PrefixIndexOracle):
    def insert(self, tokens):
        self.next_id = min(set(range(len(self.entries) + 1)) - set(self.entries))
        return super().insert(tokens)


@pytest.mark.parametrize("cls", [_ShortestMatch, _MostRecentlyUsedEviction, _FutileEviction, _HandlesReused])
def test_planted_oracle_mistake_is_caught(cls):
    class Side(OracleSide):
        def __init__(self, n_hot, max_slabs):
            self.x = cls(n_hot, max_slabs=max_slabs)
    with pytest.raises(AssertionError):
        run_scenario(Side)

"""Prefix lifecycle on the GPU: prefixes cached through the radix index (HOT first, COLD
fallback with slots shared by the prefix's requests, eviction of idle HOT prefixes), requests
attached by longest-prefix match, and decode attention for every request equal to the oracle's,
computed from the request's logical K/V (its prefix followed by its own tokens).

GraniKV (arXiv:2608.15584): "2 Related Work" (reference-counted radix index over token ids),
"B.10 Cross-pool admission and promotion policy" (HOT first, COLD fallback, no demotion)."""

import numpy as np
import pytest

from oracle import attention as OA

pytestmark = pytest.mark.gpu

N_Q, N_KV, D = 32, 8, 128


class Scene:
    def __init__(self, seed=0):
        import torch
        from shared_prefix_kv_decode_gb300 import _binding as gb
        from shared_prefix_kv_decode_gb300.cache import GraniKVCache
        self.torch = torch
        self.rng = np.random.default_rng(seed)
        self.cache = GraniKVCache(n_layers=1, n_q=N_Q, n_kv=N_KV, head_dim=D, dtype=gb.DTYPE_BF16,
                                  n_slots=20000, max_batch=32, cap=4096)
        assert self.cache.n_hot == 4000
        self.prefix = {}  # handle -> (tokens, K, V) on the host
        self.rows = []    # per active row: (tokens, K, V) logical, host float32
        self.slab = []

    def draw(self, n, scale=1.0):
        x = self.rng.standard_normal((n, N_KV, D), dtype=np.float32) * np.float32(scale)
        return self.torch.from_numpy(x).to(self.torch.bfloat16).to(self.torch.float32).numpy()

    def dev(self, x):
        return self.torch.from_numpy(np.ascontiguousarray(x)).cuda().to(self.torch.bfloat16)

    def admit(self, tokens):
        k, v = self.draw(len(tokens)), self.draw(len(tokens))
        info, evicted = self.cache.admit(tokens, [self.dev(k)], [self.dev(v)])
        self.prefix[info["prefix_id"]] = (list(tokens), k, v)
        for pid in evicted:
            del self.prefix[pid]
        return info, evicted

    def start(self, tokens):
        """A request whose prompt is `tokens`; reuses the longest cached prefix."""
        b = len(self.rows)
        slab, reused = self.cache.attach(b, tokens)
        if reused:
            pid = self.cache.row_prefix[b][0]
            ptok, pk, pv = self.prefix[pid]
            assert tokens[:reused] == ptok
            k, v = [pk], [pv]
        else:
            k, v = [], []
        own = len(tokens) - reused
        ok, ov = self.draw(own), self.draw(own)
        n_new = [0] * (b + 1)
        n_new[b] = own
        if own:
            self.cache.append(n_new, [self.dev(ok)], [self.dev(ov)])
        k.append(ok)
        v.append(ov)
        self.rows.append((tokens, np.concatenate(k), np.concatenate(v)))
        self.slab.append(slab)
        return b

    def finish(self, b):
        self.cache.detach(b)
        last = len(self.rows) - 1
        if b != last:
            self.cache.move_row(last, b)
            self.rows[b], self.slab[b] = self.rows[last], self.slab[last]
        self.rows.pop()
        self.slab.pop()

    def check_attention(self):
        torch = self.torch
        B = len(self.rows)
        q = self.rng.standard_normal((B, N_Q, D), dtype=np.float32) / np.float32(np.sqrt(D))
        q = torch.from_numpy(q).to(torch.bfloat16).to(torch.float32).numpy()
        batch = self.cache.batch(self.slab)
        o, lse = self.cache.decode(0, self.dev(q), batch)
        self.cache.ctx.sync_status(self.cache.stream())
        o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
        scale = OA.softmax_scale(D)
        for b, (_, K, V) in enumerate(self.rows):
            for h in range(N_Q):
                j = OA.kv_head(h, N_Q, N_KV)
                o_ref, lse_ref = OA.attend(q[b, h].astype(np.float64), K[:, j].astype(np.float64),
                                           V[:, j].astype(np.float64), scale)
                assert np.max(np.abs(o[b, h] - o_ref)) <= 1e-2, (b, h)
                assert abs(lse[b, h] - lse_ref) <= 1e-3, (b, h)
        return batch


def _tok(rng, base, n):
    return [int(x) for x in base + rng.integers(0, 1000, size=n)]


def test_lifecycle_hot_cold_eviction_parity(cuda_ok):
    sc = Scene(seed=5)
    rng = np.random.default_rng(11)
    p0 = _tok(rng, 0, 2500)
    p1 = _tok(rng, 10_000, 1800)
    p2 = _tok(rng, 20_000, 900)
    i0, ev = sc.admit(p0)
    assert i0["slab_id"] >= 0 and i0["slot_offset"] == 0 and not ev
    # P0 held by its requests: the next prefix (1800 > 1500 free) cannot evict it -> COLD
    for _ in range(6):
        sc.start(p0 + _tok(rng, 50_000, int(rng.integers(1, 300))))
    free_before = sc.cache.ctx.cold_free_count()
    i1, ev = sc.admit(p1)
    assert i1["slab_id"] == -1 and not ev
    assert sc.cache.ctx.cold_free_count() == free_before - 1800  # stored once
    i2, _ = sc.admit(p2)
    assert i2["slab_id"] >= 0 and i2["slot_offset"] == 2500
    rows_p1 = [sc.start(p1 + _tok(rng, 60_000, int(rng.integers(1, 300)))) for _ in range(5)]
    for _ in range(3):
        sc.start(p2 + _tok(rng, 70_000, int(rng.integers(1, 300))))
    sc.start(_tok(rng, 80_000, 700))              # no cached prefix
    sc.start(p0[:100] + _tok(rng, 90_000, 50))    # shares only part of P0: no reuse
    assert sc.slab[-1] == -1 and sc.slab[-2] == -1
    shared = sc.cache.cold_prefix_slots[i1["prefix_id"]].cpu()
    for b in rows_p1:
        assert sc.slab[b] == -1
        assert sc.torch.equal(sc.cache.req_to_slot[b, :1800].cpu(), shared)
    batch = sc.check_attention()

    # P0's requests finish: P0 is idle, and a new prefix of 2400 evicts it and takes its extent
    for b in sorted([b for b in range(len(sc.rows)) if sc.slab[b] == i0["slab_id"]], reverse=True):
        sc.finish(b)
    assert sc.cache.index.info(i0["prefix_id"])["refcount"] == 0
    p3 = _tok(rng, 30_000, 2400)
    i3, ev = sc.admit(p3)
    assert ev == [i0["prefix_id"]] and i3["slab_id"] >= 0 and i3["slot_offset"] == 0
    for _ in range(4):
        sc.start(p3 + _tok(rng, 40_000, int(rng.integers(1, 300))))
    sc.check_attention()

    # the COLD prefix's requests finish; removing it returns its 1800 slots
    for b in sorted([b for b in range(len(sc.rows)) if sc.rows[b][0][:1800] == p1], reverse=True):
        sc.finish(b)
    before = sc.cache.ctx.cold_free_count()
    sc.cache.remove_prefix(i1["prefix_id"])
    assert sc.cache.ctx.cold_free_count() == before + 1800
    sc.check_attention()
    del batch

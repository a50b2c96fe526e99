"""Multi-prefix sensitivity at kernel level: k distinct shared prefixes under one KV budget.

GraniKV (arXiv:2608.15584), "B.8 Multi-prefix sensitivity": uniform-length multi-prefix sweep
k in {1, 4, 16, 64} on the Llama-3.1-8B shape at L_p = 8K and B = 256; k = 1 is the
single-prefix case, and at k = 64 the prefixes (64 x 8K tokens) outgrow the KV working set.
Here the prefixes go through the library's prefix index as a server would admit them: prefix i
is admitted when its first requests arrive, and those requests hold it, so once HOT is full the
later prefixes are placed in COLD ("B.10 Cross-pool admission and promotion policy": HOT first,
COLD fallback, no demotion) and their requests gather them token by token from shared COLD
slots.  Requests are spread round-robin over the prefixes; each has its own log-normal suffix
(median 300, sigma 1, clipped to [32, 2048]) appended in interleaved chunks so that its COLD
slots scatter.

KV budget: the tokens that 230 GiB of HBM hold for Llama-3.1-8B (32 layers x 4 KiB per token per
layer): n_slots = 1,884,160, of which the HOT fraction 0.2 holds 46 prefixes of 8K.  One layer
of that budget is allocated and timed; the time of one decode-attention call is the median of
--reps calls, the L2 flushed before each.  K/V values come from torch's device generator (their
values do not affect the time).

  python -m shared_prefix_kv_decode_gb300.prefix_sweep [--k 1 4 16 64] [--lp 8192] [--b 256]
"""

from __future__ import annotations

import argparse
import json
import math
import statistics
import sys
from typing import Dict, List

BUDGET_SLOTS = 230 * (1 << 30) // (32 * 4096)  # 1,884,160


def build(k: int, L_p: int, B: int, n_slots: int = BUDGET_SLOTS, seed: int = 0):
    import numpy as np
    import torch
    from . import _binding as gb
    from .cache import GraniKVCache

    n_q, n_kv, d = 32, 8, 128
    rng = np.random.default_rng([seed, k])
    suffix = [int(v) for v in np.clip(np.rint(np.exp(rng.normal(math.log(300.0), 1.0, size=B))), 32, 2048)]
    cache = GraniKVCache(n_layers=1, n_q=n_q, n_kv=n_kv, head_dim=d, dtype=gb.DTYPE_BF16, n_slots=n_slots,
                         max_batch=B, cap=L_p + max(suffix) + 64)
    dev = cache.device
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)

    def rand(n):
        return torch.randn((n, n_kv, d), generator=gen, device=dev).to(torch.bfloat16)

    owner = [b % k for b in range(B)]
    slab_ids = [-1] * B
    placed: List[Dict] = []
    for i in range(k):
        tokens = [i * 1_000_000 + t for t in range(L_p)]
        info, evicted = cache.admit(tokens, [rand(L_p)], [rand(L_p)])
        assert not evicted  # every cached prefix is held by its requests
        placed.append(info)
        for b in [b for b in range(B) if owner[b] == i]:
            own_first = 1_000_000_000 + b  # a token no prefix contains
            slab, reused = cache.attach(b, tokens + [own_first])
            assert reused == L_p
            slab_ids[b] = slab
    # own suffix tokens, interleaved across requests in chunks of up to 512
    remaining = np.array(suffix, dtype=np.int64)
    while remaining.sum() > 0:
        take = np.minimum(rng.integers(1, 513, size=B), remaining)
        take[rng.random(B) < 0.25] = 0
        n = int(take.sum())
        if n == 0:
            continue
        cache.append([int(t) for t in take], [rand(n)], [rand(n)])
        remaining -= take
    q = (torch.randn((B, n_q, d), generator=gen, device=dev) / math.sqrt(d)).to(torch.bfloat16)
    batch = cache.batch(slab_ids)
    return cache, batch, q, placed, suffix


def measure(k: int, L_p: int, B: int, reps: int, flush, hbm_gbs: float, n_slots: int = BUDGET_SLOTS) -> Dict:
    import torch
    cache, batch, q, placed, suffix = build(k, L_p, B, n_slots)
    plan = cache.ctx.dispatch(batch)
    groups = plan.groups()
    stream = cache.stream()
    o, lse = cache.decode(0, q, batch, plan)
    for _ in range(2):
        cache.decode(0, q, batch, plan, o, lse)
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        cache.decode(0, q, batch, plan, o, lse)
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1) * 1000.0)
    cache.ctx.sync_status(stream)
    us = statistics.median(times)
    row = 4096  # K + V bytes of one token over 8 KV heads x 128, bf16
    n_hot = sum(1 for p in placed if p["slab_id"] >= 0)
    cold_tokens = sum(cache.seq_len_host[:B])
    alg = row * (n_hot * L_p + cold_tokens) + 4 * cold_tokens + B * 32 * 128 * 2 * 2 + B * 32 * 4
    out = {"k": k, "L_p": L_p, "B": B, "n_slots": n_slots, "hot_prefixes": n_hot,
           "cold_prefixes": k - n_hot, "suffix_tokens": sum(suffix), "cold_tokens_read": cold_tokens,
           "groups_dense": sum(1 for g in groups if g["backend"] == 1),
           "groups_cascade": sum(1 for g in groups if g["backend"] == 2),
           "us_per_call": round(us, 2), "qtok_per_s": round(B / (us * 1e-6)),
           "alg_bytes": alg, "gbs": round(alg / (us * 1e-6) / 1e9, 1),
           "frac_of_measured_hbm": round(alg / (us * 1e-6) / 1e9 / hbm_gbs, 3)}
    del cache
    torch.cuda.empty_cache()
    return out


def main(argv=None):
    import os
    import torch

    ap = argparse.ArgumentParser()
    ap.add_argument("--k", type=int, nargs="+", default=[1, 4, 16, 64])
    ap.add_argument("--lp", type=int, default=8192)
    ap.add_argument("--b", type=int, default=256)
    ap.add_argument("--reps", type=int, default=10)
    a = ap.parse_args(argv)
    torch.cuda.set_device(0)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    scratch = torch.empty((max(2 * l2, 256 << 20),), dtype=torch.uint8, device="cuda")
    peaks = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "MEASURED_PEAKS.json")
    try:
        with open(peaks) as f:
            hbm = float(json.load(f)["hbm_gbs"])
    except Exception:
        hbm = 6800.0

    def flush():
        scratch.fill_(1)

    for k in a.k:
        print(json.dumps(measure(k, a.lp, a.b, a.reps, flush, hbm)), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())

"""Contiguous HOT prefix vs. a paged-equivalent prefix, through the same library.

GraniKV (arXiv:2608.15584), "4 Experiments", kernel mechanism: the storage layout alone speeds
up the prefix attention kernel (15.6x on A100) by moving it from HBM-bound to compute-bound,
because the HOT layout reads the shared K/V once per step while a unique paged-equivalent
layout re-reads the prefix once per request.  The card page repeats the comparison.

This builds one logical batch (one shared prefix, B requests, short suffixes) twice:
  * HOT:    the prefix in one contiguous slab, the suffixes in COLD (dense or cascade backend);
  * paged:  every request carries its own copy of the prefix at the head of its COLD token
            table (the paged fallback of "B.10 Cross-pool admission and promotion policy"), so
            the prefix is gathered token by token and read B times.
Both run through granikv_decode_attention; the L2 is flushed before every timed call.

  python -m shared_prefix_kv_decode_gb300.layout_bench [--lp 16384] [--b 64] [--reps 10]
"""

from __future__ import annotations

import argparse
import json
import math
import statistics
import sys


def build(L_p: int, B: int, suffix: int, paged: bool, seed: int = 0):
    """The batch of one shared prefix of L_p tokens and B requests with `suffix` own tokens
    each, values from the seeded workload generator (``workloads.dispatch_sweep_cell``), placed
    in the HOT layout or the paged-equivalent one.  Returns (cache, batch, q, workload)."""
    import numpy as np
    import torch
    import workloads as W
    from . import _binding as gb
    from .cache import GraniKVCache

    wl = W.dispatch_sweep_cell(L_p, B, seed=seed, suffix_len=suffix)
    n_q, n_kv, d = wl.spec.n_q, wl.spec.n_kv, wl.spec.d
    cold_tokens = B * (suffix + (L_p if paged else 0))
    n_slots = max(int(math.ceil(L_p / 0.2)) + 8, int(math.ceil((cold_tokens + 1024) / 0.8)) + 8)
    cap = suffix + (L_p if paged else 0) + 64
    cache = GraniKVCache(n_layers=1, n_q=n_q, n_kv=n_kv, head_dim=d, dtype=gb.DTYPE_BF16, n_slots=n_slots,
                         max_batch=B, cap=cap)
    dev = cache.device

    def on_dev(x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(device=dev).to(torch.bfloat16)

    kp, vp = on_dev(wl.prefix_k(0)), on_dev(wl.prefix_v(0))
    ks = on_dev(np.stack([wl.suffix_k(b) for b in range(B)]))
    vs = on_dev(np.stack([wl.suffix_v(b) for b in range(B)]))
    q = on_dev(wl.q)
    if paged:
        # each request's COLD table: its private copy of the prefix, then its suffix
        for b in range(B):
            cache.append([0] * b + [L_p], [kp], [vp])
        cache.append([suffix] * B, [ks.reshape(-1, n_kv, d)], [vs.reshape(-1, n_kv, d)])
        slab_ids = [-1] * B
    else:
        sid = cache.admit_prefix(L_p, [kp], [vp])
        cache.append([suffix] * B, [ks.reshape(-1, n_kv, d)], [vs.reshape(-1, n_kv, d)])
        slab_ids = [sid] * B
    batch = cache.batch(slab_ids)
    return cache, batch, q, wl


def time_call(cache, batch, q, backend: int, reps: int, flush):
    import torch
    cache.ctx.force_backend(backend)
    plan = cache.ctx.dispatch(batch)
    o, lse = cache.decode(0, q, batch, plan)
    stream = cache.stream()
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
    return statistics.median(times), o, lse


def main(argv=None):
    import torch
    from . import _binding as gb

    ap = argparse.ArgumentParser()
    ap.add_argument("--lp", type=int, default=16384)
    ap.add_argument("--b", type=int, default=64)
    ap.add_argument("--suffix", type=int, default=256)
    ap.add_argument("--reps", type=int, default=10)
    a = ap.parse_args(argv)
    torch.cuda.set_device(0)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    scratch = torch.empty((max(2 * l2, 256 << 20),), dtype=torch.uint8, device="cuda")

    def flush():
        scratch.fill_(1)

    out = {"L_p": a.lp, "B": a.b, "suffix": a.suffix}
    cache, batch, q, _ = build(a.lp, a.b, a.suffix, paged=False)
    out["hot_dense_us"], o_d, _ = time_call(cache, batch, q, gb.BACKEND_DENSE, a.reps, flush)
    out["hot_cascade_us"], o_c, _ = time_call(cache, batch, q, gb.BACKEND_CASCADE, a.reps, flush)
    o_hot = o_d.float()
    del cache
    torch.cuda.empty_cache()
    cache, batch, q, _ = build(a.lp, a.b, a.suffix, paged=True)
    out["paged_us"], o_p, _ = time_call(cache, batch, q, gb.BACKEND_AUTO, a.reps, flush)
    out["max_abs_diff_hot_vs_paged"] = float((o_hot - o_p.float()).abs().max())
    out["speedup_dense_vs_paged"] = out["paged_us"] / out["hot_dense_us"]
    out["speedup_best_vs_paged"] = out["paged_us"] / min(out["hot_dense_us"], out["hot_cascade_us"])
    print(json.dumps(out))
    return 0


if __name__ == "__main__":
    sys.exit(main())

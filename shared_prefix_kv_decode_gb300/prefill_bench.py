"""Causal prefill of a HOT slab: time and tensor-core throughput per layer.

GraniKV (arXiv:2608.15584), "2 Related Work": a cached prefix is prefilled once and then reused
for every request that starts with it; the card page: the HOT slab holds that prefix's K_p
contiguously.  This times granikv_prefill_attention (the copy of K/V into the slab excluded)
on the Llama-3.1-8B attention shape (32/8/128, bf16) for a few prefix lengths.  Work per call:
4 * d * n_q * L_p * (L_p + 1) / 2 flops (QK^T and PV over the causal triangle); the roofline is
the measured dense bf16 tensor-core peak.  Inputs from torch's seeded device generator; the L2
is flushed before every timed call.

  python -m shared_prefix_kv_decode_gb300.prefill_bench [--lp 4096 8192 16384 32768] [--reps 5]
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys


def measure(L_p: int, reps: int, flush, peak_tflops: float, n_q: int = 32, n_kv: int = 8, d: int = 128):
    import torch
    from . import _binding as gb
    from .cache import GraniKVCache

    cache = GraniKVCache(n_layers=1, n_q=n_q, n_kv=n_kv, head_dim=d, dtype=gb.DTYPE_BF16,
                         n_slots=int(math.ceil(L_p / 0.2)) + 64, max_batch=4, cap=16)
    dev = cache.device
    gen = torch.Generator(device=dev)
    gen.manual_seed(L_p)
    q = (torch.randn((L_p, n_q, d), generator=gen, device=dev) / math.sqrt(d)).to(torch.bfloat16)
    k = torch.randn((L_p, n_kv, d), generator=gen, device=dev).to(torch.bfloat16)
    v = torch.randn((L_p, n_kv, d), generator=gen, device=dev).to(torch.bfloat16)
    sid, _ = cache.ctx.hot_alloc(L_p)
    o, lse = cache.prefill(0, sid, q, k, v)
    for _ in range(2):
        cache.prefill(0, sid, q, o=o, lse=lse)
    stream = cache.stream()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        cache.prefill(0, sid, q, o=o, lse=lse)
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1) * 1000.0)
    cache.ctx.sync_status(stream)
    us = statistics.median(times)
    flops = 4.0 * d * n_q * L_p * (L_p + 1) / 2.0
    tf = flops / (us * 1e-6) / 1e12
    del cache
    torch.cuda.empty_cache()
    return {"L_p": L_p, "n_q": n_q, "n_kv": n_kv, "d": d, "us_per_call": round(us, 1),
            "tflops": round(tf, 1), "frac_of_measured_bf16": round(tf / peak_tflops, 3)}


def main(argv=None):
    import torch
    ap = argparse.ArgumentParser()
    ap.add_argument("--lp", type=int, nargs="+", default=[4096, 8192, 16384, 32768])
    ap.add_argument("--reps", type=int, default=5)
    a = ap.parse_args(argv)
    torch.cuda.set_device(0)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    scratch = torch.empty((max(2 * l2, 256 << 20),), dtype=torch.uint8, device="cuda")
    peaks = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "MEASURED_PEAKS.json")
    try:
        with open(peaks) as f:
            peak = float(json.load(f)["bf16_tflops"])
    except Exception:
        peak = 1900.0

    def flush():
        scratch.fill_(1)

    for L_p in a.lp:
        print(json.dumps(measure(L_p, a.reps, flush, peak)), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())

"""Re-fit the dense/cascade crossover M_sat on this GPU.

GraniKV (arXiv:2608.15584), "3 GraniKV" per-step dispatch and "B.4 Per-Step Dispatch
Trace": the dispatcher runs the dense backend when M_eff = B * n_q / n_kv >= M_sat; the pages
measure M_sat = 1024 on A100 and say other GPUs need a re-fit ("Limitations").

This sweeps the Llama-3.1-8B attention shape (32/8/128, bf16; --n-q 40 for the Qwen-2.5 TP1 shape) over
L_p in {512, 2048, 8192, 16384, 32768} x B in {1, 8, 32, 128, 256, 512} with 256 COLD tokens
per request, timing decode attention with the backend forced to DENSE, forced to CASCADE, and
dispatched (AUTO).  The L2 is flushed before every timed call (or, with --layers N, before every
decode step of N back-to-back calls on N layers' own pools).  M_sat is the grid threshold whose
dispatch loses the least time against the faster backend of each cell (summed log slowdown over
the table).

  python -m shared_prefix_kv_decode_gb300.msat_fit [--reps 20] [--layers 32] [--json out.json]
"""

from __future__ import annotations

import argparse
import json
import math
import statistics
import sys

LPS = [512, 2048, 8192, 16384, 32768]
BS = [1, 8, 32, 128, 256, 512]
SUFFIX = 256


def _time_cell(L_p, B, reps, m_sat_probe, flush, gb, torch, serial=False, layers=1, suffix=SUFFIX, n_q=32,
               l2_ahead=-1, fused=False):
    """Median microseconds of one decode-attention call per backend.  layers = 1: a single call
    after an L2 flush.  layers > 1: a decode step of that many back-to-back calls, one per layer
    (each layer its own pools, so no layer's bytes are in L2 for the next), after one flush; the
    call time is the step's time over the layers.  suffix: COLD tokens per request (0: the call
    is the prefix kernel and the merge alone).  n_q: query heads (8 KV heads of 128 dims)."""
    from .cache import GraniKVCache

    n_kv, d = 8, 128
    n_cold = B * suffix + 1024
    n_slots = max(int(math.ceil(L_p / 0.2)) + 8, int(math.ceil(n_cold / 0.8)) + 8)
    cache = GraniKVCache(n_layers=layers, n_q=n_q, n_kv=n_kv, head_dim=d, dtype=gb.DTYPE_BF16, n_slots=n_slots,
                         max_batch=B, cap=suffix + 64)
    dev = cache.device
    gen = torch.Generator(device=dev)
    gen.manual_seed(L_p * 1000 + B)
    k = torch.randn((L_p, n_kv, d), generator=gen, device=dev).to(torch.bfloat16)
    v = torch.randn((L_p, n_kv, d), generator=gen, device=dev).to(torch.bfloat16)
    sid = cache.admit_prefix(L_p, [k] * layers, [v] * layers)
    if suffix > 0:
        kn = torch.randn((B * suffix, n_kv, d), generator=gen, device=dev).to(torch.bfloat16)
        vn = torch.randn((B * suffix, n_kv, d), generator=gen, device=dev).to(torch.bfloat16)
        cache.append([suffix] * B, [kn] * layers, [vn] * layers)
    q = (torch.randn((B, n_q, d), generator=gen, device=dev) / math.sqrt(d)).to(torch.bfloat16)
    batch = cache.batch([sid] * B)
    if serial:  # prefix, suffix and merge one after another, each kernel on all SMs
        cache.ctx.set_concurrency(False, 0.0)
    cache.ctx.set_dense_l2_ahead(l2_ahead)
    cache.ctx.set_fused_merge(fused)
    out = {}
    stream = cache.stream()
    names = (("dense", gb.BACKEND_DENSE), ("cascade", gb.BACKEND_CASCADE), ("auto", gb.BACKEND_AUTO))
    plans, outs = {}, {}
    for name, backend in names:
        cache.ctx.force_backend(backend)
        plans[name] = cache.ctx.dispatch(batch, cache.ctx.plan())
        outs[name] = cache.decode(0, q, batch, plans[name])
        out[name + "_backend"] = gb.BACKEND_NAMES[plans[name].groups()[0]["backend"]]
    torch.cuda.synchronize()
    # the three plans take turns within every repetition, so that slow drift of the GPU's
    # state is not read as a difference between them, and the turn order rotates from one
    # repetition to the next, so that no plan always runs after the same one
    times = {name: [] for name, _ in names}
    for rep in range(reps):
        for name, _ in names[rep % len(names):] + names[:rep % len(names)]:
            o, lse = outs[name]
            flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for layer in range(layers):
                cache.decode(layer, q, batch, plans[name], o, lse)
            e1.record(stream)
            e1.synchronize()
            times[name].append(e0.elapsed_time(e1) * 1000.0 / layers)
    for name, _ in names:
        out[name] = statistics.median(times[name])
    cache.ctx.sync_status(stream)
    return out


def fit_msat(rows, g=4):
    """The threshold that fits the measured table best: among the grid's M_eff values (and one
    past the largest, i.e. cascade everywhere), the M_sat whose dispatch (dense at M_eff >= M_sat,
    cascade below) has the smallest summed log slowdown against the faster backend of each cell.
    Ties go to the larger M_sat.  A single noisy cell thus moves the threshold only when it
    outweighs the cells on the other side."""
    meffs = sorted({r["B"] * g for r in rows})
    cands = meffs + [2 * meffs[-1]]

    def regret(m_sat):
        tot = 0.0
        for r in rows:
            t = r["dense_us"] if r["B"] * g >= m_sat else r["cascade_us"]
            tot += math.log(t / min(r["dense_us"], r["cascade_us"]))
        return tot

    return min(cands, key=lambda m: (round(regret(m), 12), -m))


def fit_msat_strict(rows, g=4, min_lp=2048):
    """The stricter reading: the smallest grid M_eff from which on the dense backend is no
    slower than the cascade one at every L_p >= min_lp (that M_eff and every larger one); one
    past the largest M_eff when no such value exists."""
    meffs = sorted({r["B"] * g for r in rows})
    for m in meffs:
        if all(r["dense_us"] <= r["cascade_us"] for r in rows if r["B"] * g >= m and r["L_p"] >= min_lp):
            return m
    return 2 * meffs[-1]


def dispatch_ratio(row):
    """Dispatched time over the faster single backend's, for one measured cell."""
    return row["auto_us"] / min(row["dense_us"], row["cascade_us"])


def main(argv=None):
    import torch
    from . import _binding as gb

    ap = argparse.ArgumentParser()
    ap.add_argument("--reps", type=int, default=15)
    ap.add_argument("--json", default=None)
    ap.add_argument("--lps", default=",".join(map(str, LPS)))
    ap.add_argument("--bs", default=",".join(map(str, BS)))
    ap.add_argument("--serial", action="store_true", help="run each kernel on its own (for profiling)")
    ap.add_argument("--layers", type=int, default=1,
                    help="time decode steps of this many back-to-back layer calls (default: single calls)")
    ap.add_argument("--n-q", type=int, default=32, help="query heads (40: the Qwen-2.5 TP1 shape)")
    ap.add_argument("--fused-merge", action="store_true",
                    help="merge each row in the producer that finishes it last (no merge kernel)")
    ap.add_argument("--dense-l2-ahead", type=int, default=-1,
                    help="dense kernel's L2 read-ahead in tiles (-1: the library's per-step choice)")
    ap.add_argument("--suffix", type=int, default=SUFFIX,
                    help="COLD tokens per request (0: time the prefix kernel and the merge alone)")
    a = ap.parse_args(argv)
    torch.cuda.set_device(0)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    scratch = torch.empty((max(2 * l2, 256 << 20),), dtype=torch.uint8, device="cuda")

    def flush():
        scratch.fill_(1)

    rows = []
    for L_p in [int(x) for x in a.lps.split(",")]:
        for B in [int(x) for x in a.bs.split(",")]:
            r = _time_cell(L_p, B, a.reps, None, flush, gb, torch, serial=a.serial, layers=a.layers,
                           suffix=a.suffix, n_q=a.n_q, l2_ahead=a.dense_l2_ahead, fused=a.fused_merge)
            row = {"L_p": L_p, "B": B, "m_eff": B * a.n_q // 8, "dense_us": r["dense"], "cascade_us": r["cascade"],
                   "auto_us": r["auto"], "auto_backend": r["auto_backend"]}
            rows.append(row)
            print(json.dumps(row), flush=True)
            torch.cuda.empty_cache()
    m_sat = fit_msat(rows, g=a.n_q // 8)
    m_strict = fit_msat_strict(rows, g=a.n_q // 8)
    worst = max(rows, key=dispatch_ratio)
    print(f"# fitted M_sat = {m_sat} (least regret); strict rule: {m_strict}; "
          f"worst dispatched / best backend: {dispatch_ratio(worst):.3f} at L_p {worst['L_p']} B {worst['B']}")
    print("| L_p | B | M_eff | dense us | cascade us | auto us | auto -> | best/auto |")
    print("|---|---|---|---|---|---|---|---|")
    for r in rows:
        best = min(r["dense_us"], r["cascade_us"])
        print(f"| {r['L_p']} | {r['B']} | {r['m_eff']} | {r['dense_us']:.1f} | {r['cascade_us']:.1f} | "
              f"{r['auto_us']:.1f} | {r['auto_backend']} | {best / r['auto_us']:.3f} |")
    if a.json:
        with open(a.json, "w") as f:
            json.dump({"rows": rows, "m_sat": m_sat, "m_sat_strict": m_strict, "layers": a.layers, "reps": a.reps,
                       "suffix": a.suffix}, f, indent=1)
    return 0


if __name__ == "__main__":
    sys.exit(main())

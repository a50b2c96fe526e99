#!/usr/bin/env python3
"""Decode-step attention benchmark for GraniKV's HOT/COLD KV cache on GB300.

Metric: decode-attention query-tokens/s (one decode query token per request per layer) on
the Llama-3.1-8B attention shape with one shared prefix of L_p = 16384 tokens, B = 64
requests and log-normal suffixes (median 300), plus the achieved fraction of the HBM
roofline of the decode-attention launches.

A step is one pass of the whole path over one batch: COLD slot allocation for one new token
per request, the scatter of each layer's new K/V into the COLD pool, the per-step dispatch,
and decode attention (prefix partial, suffix partial, log-sum-exp merge) for every layer.
Each layer has its own K/V pools, so one step touches far more memory than the 129 MB L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--layers L] [--impl granikv|reference]

Under torchrun (N > 1) every rank runs an independent replica (request-level data
parallelism, no collective on the data path); rank 0 prints one JSON line with the whole-job
throughput over the slowest rank's time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn query-tokens/s at L_p=16K on 1 GB300; % HBM / tensor roofline"
UNIT = "q-tok/s"
WORKLOAD = "llama8b_single_prefix_16k"  # the headline configuration
# Other full-size configurations the bench can run (``--workload``); the headline line is the
# default one.
WORKLOADS = {  # name -> suffix description
    "llama8b_single_prefix_16k": (None, "log-normal median 300, sigma 1, clipped [32, 2048]"),
    "hetero_multi_prefix_k8": (None, "8 prefixes L_p ~ U[2048, 16384], 8-32 requests each, log-normal suffixes"),
    "qwen_tp1_16k": (None, "suffix U[64, 1024]"),
}
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--layers", type=int, default=32)
    ap.add_argument("--impl", choices=["granikv", "reference"], default="granikv")
    ap.add_argument("--backend", choices=["auto", "dense", "cascade"], default="auto")
    ap.add_argument("--serial", action="store_true",
                    help="run the prefix and suffix kernels one after the other on the caller's stream")
    ap.add_argument("--prefix-share", type=float, default=0.0,
                    help="share of the SMs the prefix work list is sized for when running concurrently "
                         "(0: the library's automatic share)")
    ap.add_argument("--fused-merge", action="store_true",
                    help="merge each row in the producer that finishes it last (no merge kernel)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fused-append", action="store_true",
                    help="append each layer's new K/V with its own launch before the attention call")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=WORKLOAD,
                    help="full-size configuration to time (default: the headline one)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="rough bound on the CPU-baseline sample's run time")
    return ap.parse_args(argv)


# ---- distributed plumbing (host-side timing reduction only) --------------------------------

def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a host scalar over all ranks (no-op for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---- accounting -----------------------------------------------------------------------------

def workload_fn(name):
    import workloads as W
    return {"llama8b_single_prefix_16k": W.llama8b_single_prefix_16k,
            "hetero_multi_prefix_k8": W.hetero_multi_prefix_k8,
            "qwen_tp1_16k": W.qwen_tp1_16k}[name]


def algorithmic_bytes(spec, slab_ids, seq_lens, esize: int) -> int:
    """Bytes one decode-attention call must move at minimum: each HOT prefix's K and V once,
    every COLD token's K and V plus its 4-byte table entry, q and o once, lse once."""
    row = spec.n_kv * spec.d * esize
    prefixes = {s for s in slab_ids if s >= 0}
    lp_of = {}
    for b, s in enumerate(slab_ids):
        if s >= 0:
            lp_of[s] = spec.prefix_lens[spec.req_prefix[b]]
    prefix = sum(2 * lp_of[s] * row for s in prefixes)
    cold = sum(2 * L * row + 4 * L for L in seq_lens)
    B = len(seq_lens)
    qo = 2 * B * spec.n_q * spec.d * esize + 4 * B * spec.n_q
    return prefix + cold + qo


def algorithmic_flops(spec, slab_ids, seq_lens) -> int:
    tot = 0
    for b, s in enumerate(slab_ids):
        lp = spec.prefix_lens[spec.req_prefix[b]] if s >= 0 else 0
        tot += 4 * spec.d * spec.n_q * (lp + seq_lens[b])
    return tot


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def source_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "shared_prefix_kv_decode_gb300", "csrc")
    for n in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(n.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_tag: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel and workload, if it
    was taken on the current sources; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.md")
    if not os.path.exists(path):
        return None
    digest = None
    traffic = None
    with open(path) as f:
        for line in f:
            if line.startswith("source_digest:"):
                digest = line.split(":", 1)[1].strip()
            if line.startswith("dram_bytes_per_launch:"):
                try:
                    traffic = float(line.split(":", 1)[1].strip())
                except ValueError:
                    traffic = None
    if digest != source_digest():
        return None
    return traffic


# ---- clocks ------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str):
        self.uuid = uuid
        self.proc = None
        self.path = os.path.join("/tmp", f"granikv_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "10"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        all_rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    all_rows.append(parts)
        rows = [r for r in all_rows if self.uuid and self.uuid in r[0]]
        if not rows and len({r[0] for r in all_rows}) == 1:
            rows = all_rows
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        busy = [x for x in sm if mx and x > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ---- CPU baseline (the oracle, as it stands) -------------------------------------------------

def cpu_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def host_cores_note() -> str:
    try:
        aff = len(os.sched_getaffinity(0))
    except Exception:
        aff = None
    return f"os.cpu_count()={os.cpu_count()}, affinity {aff}, BLAS threads {cpu_threads()}"


def oracle_sample(wl, requests):
    import oracle.attention as OA
    t = time.perf_counter()
    for b in requests:
        OA.request_attention(wl, b)
    return time.perf_counter() - t


def cpu_baseline(wl, seconds: float):
    """Time the fp64 oracle on a bounded sample of the workload's requests (one layer)."""
    B = wl.spec.B
    t1 = oracle_sample(wl, [0])
    n = max(1, min(B, int(seconds / max(t1, 1e-6))))
    reqs = list(range(n))
    t = oracle_sample(wl, reqs)
    return {"value": n / t, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
            "sample": f"{n} of {B} requests of {wl.spec.name}, one layer, fp64 numpy oracle "
                      f"({t:.1f} s; host cores: {host_cores_note()})"}


# ---- the reference arm: the oracle on the host cores ----------------------------------------

def run_reference(args):
    world, rank, local = dist_info()
    if rank != 0:
        return 0
    import workloads as W
    wl = workload_fn(args.workload)(seed=0)
    per_step = 2
    B = wl.spec.B
    for i in range(args.warmup):
        oracle_sample(wl, [(i * per_step + k) % B for k in range(per_step)])
    times = []
    for i in range(args.steps):
        times.append(oracle_sample(wl, [((args.warmup + i) * per_step + k) % B for k in range(per_step)]))
    t = sum(times)
    value = per_step * args.steps / t
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000.0 * t / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": args.workload, "n_q": wl.spec.n_q, "n_kv": wl.spec.n_kv,
                       "head_dim": wl.spec.d, "L_p": wl.spec.prefix_lens[0],
                       "B": B, "sample_per_step": f"{per_step} requests, one layer"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                             "sample": f"{per_step} requests per step of {wl.spec.name}, one layer "
                                       f"(host cores: {host_cores_note()})"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---- the GraniKV arm -------------------------------------------------------------------------

def run_granikv(args):
    import numpy as np
    import torch

    world, rank, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    import __graft_entry__
    __graft_entry__.build()
    import workloads as W
    from shared_prefix_kv_decode_gb300 import _binding as gb
    from shared_prefix_kv_decode_gb300.workload_io import load_workload

    L = args.layers
    steps_total = args.warmup + args.steps
    e2e_steps = max(3, args.steps)  # as many steps as the device-timed leg
    wl = workload_fn(args.workload)(seed=rank)
    spec = wl.spec
    B = spec.B
    extra = steps_total + e2e_steps + 8
    cap = max(wl.cold_len(b) for b in range(B)) + extra + 64
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000 + rank)

    def layer_fill(layer, shape):
        return torch.randn(shape, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)

    lw = load_workload(wl, n_layers=L, device=dev.index, cap=cap, layer_fill=layer_fill)
    cache = lw.cache
    ctx = cache.ctx
    ctx.force_backend({"auto": gb.BACKEND_AUTO, "dense": gb.BACKEND_DENSE,
                       "cascade": gb.BACKEND_CASCADE}[args.backend])
    ctx.set_checks(True)
    ctx.set_concurrency(not args.serial, args.prefix_share)
    ctx.set_fused_merge(args.fused_merge)
    stream = torch.cuda.current_stream(dev)
    # A step's inputs (q, new K, new V of every layer) live in one device buffer and its outputs
    # (o, lse of every layer) in another, so the end-to-end run moves each direction with one
    # copy per step; the per-layer tensors are views into them.
    # Two such buffer sets: the end-to-end leg copies step k+1's inputs in (and step k's outputs
    # out) on a copy stream while step k computes.
    n_qe, n_kve = B * spec.n_q * spec.d, B * spec.n_kv * spec.d
    o_bytes, l_bytes = B * spec.n_q * spec.d * 2, B * spec.n_q * 4

    def buffer_set():
        in_dev = torch.empty((L, n_qe + 2 * n_kve), dtype=torch.bfloat16, device=dev)
        out_dev = torch.empty((L, o_bytes + l_bytes), dtype=torch.uint8, device=dev)
        return {"in": in_dev, "out": out_dev,
                "q": [in_dev[layer, :n_qe].view(B, spec.n_q, spec.d) for layer in range(L)],
                "k": [in_dev[layer, n_qe:n_qe + n_kve].view(B, spec.n_kv, spec.d) for layer in range(L)],
                "v": [in_dev[layer, n_qe + n_kve:].view(B, spec.n_kv, spec.d) for layer in range(L)],
                "o": [out_dev[layer, :o_bytes].view(torch.bfloat16).view(B, spec.n_q, spec.d) for layer in range(L)],
                "lse": [out_dev[layer, o_bytes:].view(torch.float32).view(B, spec.n_q) for layer in range(L)]}

    bufs = [buffer_set(), buffer_set()]
    qs, knew, vnew = bufs[0]["q"], bufs[0]["k"], bufs[0]["v"]
    qs[0].copy_(lw.q)
    for layer in range(1, L):
        qs[layer].copy_((torch.randn((B, spec.n_q, spec.d), generator=gen, device=dev) / math.sqrt(spec.d)))
    for layer in range(L):
        knew[layer].copy_(torch.randn((B, spec.n_kv, spec.d), generator=gen, device=dev))
        vnew[layer].copy_(torch.randn((B, spec.n_kv, spec.d), generator=gen, device=dev))
    bufs[1]["in"].copy_(bufs[0]["in"])
    slots = torch.empty((B,), dtype=torch.int32, device=dev)
    plan = ctx.plan()
    slab_ids = lw.slab_ids
    seq = list(cache.seq_len_host[:B])
    # workspace sized for the largest plan of the run: suffixes grow by one token per step, and
    # the dispatcher's prefix/suffix split (so the record count) may change with them
    ws_bytes = 0
    for k in range(1, extra + 1):
        probe = gb.Batch(slab_ids, [x + k for x in seq], cache.req_to_slot, cache.cap)
        ws_bytes = max(ws_bytes, ctx.workspace_size(ctx.dispatch(probe, plan)))
    ws = torch.empty((ws_bytes,), dtype=torch.uint8, device=dev)
    ones = [1] * B
    # the COLD append fused into the attention launches
    fused = not args.no_fused_append
    ev_pairs = []
    timed_bytes = []

    def step(record, bs=0):
        bset = bufs[bs]
        ctx.cold_alloc(ones, cache.req_to_slot, cache.suffix_len, cache.cap, slots, stream)
        for i in range(B):
            seq[i] += 1
        if not fused:
            for layer in range(L):
                ctx.cold_append(layer, bset["k"][layer], bset["v"][layer], slots, B, stream)
        batch = gb.Batch(slab_ids, seq, cache.req_to_slot, cache.cap)
        ctx.dispatch(batch, plan)
        nbytes = algorithmic_bytes(spec, slab_ids, seq, 2)
        # events bracket the step's L back-to-back decode-attention calls (not each call, so
        # that nothing sits between two calls' kernels on the stream)
        if record:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
        for layer in range(L):
            if fused:  # the layer's new K/V are written to their slots by the attention launch
                ctx.decode_attention_append(layer, bset["q"][layer], bset["k"][layer], bset["v"][layer], batch, plan,
                                            bset["o"][layer], bset["lse"][layer], ws, ws_bytes, stream)
            else:
                ctx.decode_attention(layer, bset["q"][layer], batch, plan, bset["o"][layer], bset["lse"][layer], ws,
                                     ws_bytes, stream)
        if record:
            e1.record(stream)
            ev_pairs.append((e0, e1))
            timed_bytes.append(nbytes)
        return batch

    for _ in range(args.warmup):
        step(False)
    ctx.sync_status(stream)
    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", "") or "")
    sampler = ClockSampler(uuid)
    k0, c0 = ctx.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        step(True)
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier(world)
    k1, c1 = ctx.launch_count()
    ctx.sync_status(stream)
    t_local = t_start.elapsed_time(t_end) / 1000.0
    t_max = max_over_ranks(t_local, world, dev)
    value = world * B * L * args.steps / t_max
    call_ms = [a.elapsed_time(b) / L for a, b in ev_pairs]
    avg_call_s = statistics.mean(call_ms) / 1000.0
    avg_bytes = statistics.mean(timed_bytes)

    # end to end through the C ABI with host buffers: every step's inputs are copied in from
    # pinned host memory and its outputs read back inside the timed region; the copies run on a
    # copy stream, step k+1's inputs and step k's outputs while step k computes (two buffer sets)
    in_host = bufs[0]["in"].cpu().pin_memory()
    out_host = torch.empty(bufs[0]["out"].shape, dtype=bufs[0]["out"].dtype).pin_memory()
    h2d = in_host.numel() * in_host.element_size()
    d2h = out_host.numel() * out_host.element_size()
    copy_stream = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event(), torch.cuda.Event()]
    ev_done = [torch.cuda.Event(), torch.cuda.Event()]
    ev_out = [torch.cuda.Event(), torch.cuda.Event()]

    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)
    with torch.cuda.stream(copy_stream):
        bufs[0]["in"].copy_(in_host, non_blocking=True)
    ev_in[0].record(copy_stream)
    for k in range(e2e_steps):
        bs = k % 2
        stream.wait_event(ev_in[bs])
        if k >= 2:
            stream.wait_event(ev_out[bs])  # step k-2's outputs have left this set
        step(False, bs)
        ev_done[bs].record(stream)
        with torch.cuda.stream(copy_stream):
            if k + 1 < e2e_steps:
                if k >= 1:
                    copy_stream.wait_event(ev_done[1 - bs])  # step k-1 finished with that set
                bufs[1 - bs]["in"].copy_(in_host, non_blocking=True)
                ev_in[1 - bs].record(copy_stream)
            copy_stream.wait_event(ev_done[bs])
            out_host.copy_(bufs[bs]["out"], non_blocking=True)
            ev_out[bs].record(copy_stream)
    stream.wait_stream(copy_stream)
    e1.record(stream)
    torch.cuda.synchronize()
    t_e2e = max_over_ranks(e0.elapsed_time(e1) / 1000.0, world, dev)
    ctx.sync_status(stream)
    e2e_value = world * B * L * e2e_steps / t_e2e

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    hbm, tflops, peak_src = read_peaks()
    achieved = avg_bytes / avg_call_s / 1e9
    groups = plan.groups()
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": profiled_traffic("decode_attention_" + args.workload),
                "kernel": "granikv_decode_attention launches (prefix + suffix + merge)",
                "peak_source": f"{peak_src} hbm_gbs",
                "algorithmic_bytes_per_launch": avg_bytes,
                "avg_launch_us": avg_call_s * 1e6,
                "prefix_tflops": algorithmic_flops(spec, slab_ids, seq) / avg_call_s / 1e12}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1000.0 * t_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "n_q": spec.n_q, "n_kv": spec.n_kv, "head_dim": spec.d,
                   "L_p": spec.prefix_lens[0] if len(spec.prefix_lens) == 1 else list(spec.prefix_lens), "B": B,
                   "suffix": WORKLOADS[args.workload][1],
                   "layers_per_step": L, "backend": args.backend,
                   "append": "fused into the attention launch" if fused else "own launch per layer",
                   "schedule": dict(plan.schedule(), dense_l2_ahead=plan.dense_l2_ahead()),
                   "concurrency": "serial" if args.serial else f"prefix share {args.prefix_share}",
                   "merge": "by the last producer of each row" if args.fused_merge else "merge kernel",
                   "groups": [{"m_eff": g["m_eff"], "backend": gb.BACKEND_NAMES[g["backend"]],
                               "n_splits": g["n_splits"]} for g in groups],
                   "l2": (f"inputs larger than L2: each step reads {L} distinct layers' pools, "
                          f"{L * avg_bytes / 1e6:.0f} MB > 129 MB L2"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roofline,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": k1 - k0,
        "host_copies": c1 - c0,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_granikv(args)


if __name__ == "__main__":
    sys.exit(main())

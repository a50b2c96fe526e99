"""Multi-step decode driver: requests arrive and complete between steps, and every step runs the
whole decode path through the library for the realized batch.

GraniKV (arXiv:2608.15584), "3 GraniKV": the dispatcher decides per step, for the batch that is
actually running, whether a prefix group goes to the dense or the cascade backend;
"B.4 Per-Step Dispatch Trace" reports that decision step by step and "B.5 Per-Step Dispatch
Overhead" its host cost.  A step here is, for every active request:
  1. one COLD slot (granikv_cold_alloc, n_new = 1) and the new token's K/V in every layer
     (granikv_cold_append);
  2. granikv_dispatch on the realized batch (grouped by HOT slab, M_eff = B_g * n_q / n_kv);
  3. granikv_decode_attention in every layer.
Arrivals append a prompt suffix for a new request sharing one of the HOT prefixes; completions
return the request's COLD slots (granikv_cold_free) and move the last request's token table into
its row, so the active requests always occupy table rows 0..B-1.

The per-step trace holds B, the groups (M_eff, backend, pieces), the host time of the dispatch
call, the host time to issue the whole step and the GPU time of the step's attention calls.

Graph mode ("B.5 Per-Step Dispatch Overhead": the per-step host work must stay small; "B.2 Full
ShareGPT Lp x B matrix": the serving engine runs decode steps from pre-allocated CUDA graphs):
the step's slot allocation (granikv_cold_alloc_uniform) and attention calls of every layer (the
new K/V written by them, or by granikv_cold_append where that path is not available) are
captured once in a CUDA graph and replayed step after step.  The plan is made for the
requests' lengths plus a headroom and the kernels read the lengths that exist from the device
(granikv_batch.seq_len_dev), so one capture serves until the batch changes or a request would
outgrow its planned length; then the step runs eagerly once (which also uploads the new plan)
and is captured again.

  python -m shared_prefix_kv_decode_gb300.decode_driver [--steps 64] [--layers 2] [--seed 0] [--graph]
"""

from __future__ import annotations

import argparse
import json
import math
import statistics
import sys
import time
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

from . import _binding as gb
from .cache import GraniKVCache


class DecodeDriver:
    """Requests sharing HOT prefixes, decoded step by step with arrivals and completions.

    keep_logical: keep every request's logical K/V and the last step's q on the host (float32),
    so that a test can recompute the attention without reading the pools."""

    def __init__(self, *, prefix_lens: Sequence[int], n_layers: int = 1, n_q: int = 32, n_kv: int = 8,
                 head_dim: int = 128, max_batch: int = 256, cap: int = 4096, n_slots: int = 1 << 17,
                 seed: int = 0, keep_logical: bool = False, device: int = 0, graph: bool = False,
                 headroom: int = 16, fused_append: bool = True):
        self.n_layers, self.n_q, self.n_kv, self.d = n_layers, n_q, n_kv, head_dim
        self.rng = np.random.default_rng(seed)
        self.keep = keep_logical
        self.cache = GraniKVCache(n_layers=n_layers, n_q=n_q, n_kv=n_kv, head_dim=head_dim, dtype=gb.DTYPE_BF16,
                                  n_slots=n_slots, max_batch=max_batch, cap=cap, device=device)
        self.dev = self.cache.device
        self.ctx = self.cache.ctx
        self.plan = self.ctx.plan()
        self.slabs: List[int] = []
        self.prefix_kv: List[List[np.ndarray]] = []  # per prefix: [K_l, V_l] per layer (float32)
        for L_p in prefix_lens:
            k = [self._draw((L_p, n_kv, head_dim)) for _ in range(n_layers)]
            v = [self._draw((L_p, n_kv, head_dim)) for _ in range(n_layers)]
            sid = self.cache.admit_prefix(L_p, [self._dev(x) for x in k], [self._dev(x) for x in v])
            if sid is None:
                raise RuntimeError(f"no HOT space for a prefix of {L_p} tokens")
            self.slabs.append(sid)
            self.prefix_kv.append([k, v] if keep_logical else [])
        self.rows: List[Dict] = []       # active requests, row b of the token table
        self.next_id = 0
        self.trace: List[Dict] = []
        self._events = []
        self.last_q: Optional[List[np.ndarray]] = None
        self.last_out = None
        # graph mode: fixed device buffers the captured step reads and writes
        self.graph_mode, self.headroom = graph, headroom
        self.fused = fused_append and self.cache.fused_append  # new K/V written by the attention launch
        self._graph = None
        self._graph_key = None
        self._planned: List[int] = []
        self._cold_dirty = False  # graph work moved the ring position on the device only
        if graph:
            dt, dev = torch.bfloat16, self.dev
            self._q_buf = [torch.zeros((max_batch, n_q, head_dim), dtype=dt, device=dev) for _ in range(n_layers)]
            self._k_buf = [torch.zeros((max_batch, n_kv, head_dim), dtype=dt, device=dev) for _ in range(n_layers)]
            self._v_buf = [torch.zeros((max_batch, n_kv, head_dim), dtype=dt, device=dev) for _ in range(n_layers)]
            self._o_buf = [torch.zeros((max_batch, n_q, head_dim), dtype=dt, device=dev) for _ in range(n_layers)]
            self._lse_buf = [torch.zeros((max_batch, n_q), dtype=torch.float32, device=dev) for _ in range(n_layers)]
            self._slots_buf = torch.zeros((max_batch,), dtype=torch.int32, device=dev)

    # ---- helpers -------------------------------------------------------------------------
    def _draw(self, shape, scale: float = 1.0) -> np.ndarray:
        # bf16-representable float32 values, so the host copy equals what the device holds
        x = self.rng.standard_normal(shape, dtype=np.float32) * np.float32(scale)
        return torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()

    def _dev(self, x: np.ndarray) -> torch.Tensor:
        return torch.from_numpy(np.ascontiguousarray(x)).to(self.dev).to(torch.bfloat16)

    @property
    def B(self) -> int:
        return len(self.rows)

    def _sync_cold(self):
        """Bring the host's copy of the COLD ring position up to date after graph work."""
        if self._cold_dirty:
            self.ctx.cold_sync(self.cache.stream())
            self._cold_dirty = False

    def _draw_new(self, N: int):
        """K/V of N new tokens in every layer: host copies (float32) and device tensors."""
        ks = [self._draw((N, self.n_kv, self.d)) for _ in range(self.n_layers)]
        vs = [self._draw((N, self.n_kv, self.d)) for _ in range(self.n_layers)]
        return ks, vs, [self._dev(x) for x in ks], [self._dev(x) for x in vs]

    def _keep_new(self, n_new: List[int], ks, vs):
        if self.keep:
            off = 0
            for b, n in enumerate(n_new):
                r = self.rows[b]
                for layer in range(self.n_layers):
                    r["k"][layer].append(ks[layer][off:off + n])
                    r["v"][layer].append(vs[layer][off:off + n])
                off += n

    def _append(self, n_new: List[int]):
        """n_new[b] new tokens for active request b, K/V drawn here, in every layer."""
        self._sync_cold()
        ks, vs, kd, vd = self._draw_new(int(sum(n_new)))
        self.cache.append(n_new, kd, vd)
        self._keep_new(n_new, ks, vs)

    # ---- arrivals and completions --------------------------------------------------------
    def arrive(self, prefix: int, prompt_len: int):
        """A new request on HOT prefix `prefix` whose prompt suffix has prompt_len tokens."""
        if self.B >= self.cache.max_batch:
            raise RuntimeError("batch is full")
        self.rows.append({"id": self.next_id, "prefix": prefix, "len": 0,
                          "k": [[] for _ in range(self.n_layers)], "v": [[] for _ in range(self.n_layers)]})
        self.next_id += 1
        n_new = [0] * self.B
        n_new[-1] = prompt_len
        self._append(n_new)
        self.rows[-1]["len"] = prompt_len

    def complete(self, b: int):
        """Request in row b finishes: its COLD slots go back to the free list, and the last row's
        request moves into row b."""
        self._sync_cold()
        s = self.cache.stream()
        L = self.rows[b]["len"]
        if L:
            slots = self.cache.req_to_slot[b, :L].clone()
            self.ctx.cold_free(slots, L, s)
        last = self.B - 1
        if b != last:
            self.cache.req_to_slot[b].copy_(self.cache.req_to_slot[last])
            self.cache.suffix_len[b].copy_(self.cache.suffix_len[last])
            self.rows[b] = self.rows[last]
            self.cache.seq_len_host[b] = self.cache.seq_len_host[last]
        self.rows.pop()
        self.cache.seq_len_host[last] = 0
        self.cache.suffix_len[last].zero_()

    # ---- one decode step -----------------------------------------------------------------
    def step(self):
        """One decode step of every active request: one new token each (slot, K/V in every
        layer), then attention in every layer."""
        B = self.B
        if B == 0:
            return None
        for r in self.rows:
            r["len"] += 1
        slab_ids = [self.slabs[r["prefix"]] for r in self.rows]
        # the step's synthetic inputs, drawn and uploaded before the timed region
        ks, vs, kd, vd = self._draw_new(B)
        qs = [self._draw((B, self.n_q, self.d), 1.0 / math.sqrt(self.d)) for _ in range(self.n_layers)]
        q_dev = [self._dev(x) for x in qs]
        s = self.cache.stream()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if self.graph_mode:
            rec = self._step_graph(B, slab_ids, kd, vd, q_dev, e0, e1)
            out = (self._o_buf[-1][:B], self._lse_buf[-1][:B])
        else:
            self._sync_cold()
            fused = self.fused
            e0.record(s)
            t_issue = time.perf_counter()
            if fused:  # slots now, the K/V rows written by the attention launches
                self.cache.alloc([1] * B)
            else:
                self.cache.append([1] * B, kd, vd)
            batch = self.cache.batch(slab_ids, [r["len"] for r in self.rows])
            t0 = time.perf_counter()
            self.ctx.dispatch(batch, self.plan)
            t_disp = time.perf_counter() - t0
            out = None
            for layer in range(self.n_layers):
                out = self.cache.decode(layer, q_dev[layer], batch, self.plan,
                                        k_new=kd[layer] if fused else None, v_new=vd[layer] if fused else None)
            t_host = time.perf_counter() - t_issue
            e1.record(s)
            rec = {"dispatch_us": t_disp * 1e6, "host_us": t_host * 1e6, "mode": "eager"}
        self._keep_new([1] * B, ks, vs)
        self._events.append((e0, e1))
        groups = self.plan.groups()
        rec.update({"B": B, "concurrent": self.plan.schedule()["concurrent"], "groups": [{"m_eff": g["m_eff"], "backend": gb.BACKEND_NAMES[g["backend"]],
                                        "n_splits": g["n_splits"]} for g in groups]})
        self.trace.append(rec)
        if self.keep:
            self.last_q = qs
        self.last_out = out
        return out

    def _step_graph(self, B, slab_ids, kd, vd, q_dev, e0, e1) -> Dict:
        """The step as one CUDA-graph replay; re-plan and capture when the batch changed or a
        request would outgrow its planned length."""
        s = self.cache.stream()
        for layer in range(self.n_layers):
            self._k_buf[layer][:B].copy_(kd[layer])
            self._v_buf[layer][:B].copy_(vd[layer])
            self._q_buf[layer][:B].copy_(q_dev[layer])
        lens = [r["len"] for r in self.rows]  # after this step's token
        key = (B, tuple(slab_ids))
        if self._graph is not None and key == self._graph_key and all(
                n <= m for n, m in zip(lens, self._planned)):
            e0.record(s)
            t0 = time.perf_counter()
            self._graph.replay()
            t_host = time.perf_counter() - t0
            e1.record(s)
            self._cold_dirty = True
            for b in range(B):
                self.cache.seq_len_host[b] += 1
            return {"dispatch_us": 0.0, "host_us": t_host * 1e6, "mode": "replay"}
        # re-plan for the lengths plus a headroom, run this step eagerly (uploading the plan),
        # then capture the same calls for the steps to come
        self._sync_cold()
        self._planned = [min(self.cache.cap, n + self.headroom) for n in lens]
        batch = gb.Batch(slab_ids, self._planned, self.cache.req_to_slot, self.cache.cap,
                         seq_len_dev=self.cache.suffix_len)
        self._graph_batch = batch  # keeps the host arrays the captured calls point to alive
        t0 = time.perf_counter()
        self.ctx.dispatch(batch, self.plan)
        t_disp = time.perf_counter() - t0
        ws = self.cache.workspace(self.plan)

        fused = self.fused

        def issue():
            st = torch.cuda.current_stream(self.dev)
            self.ctx.cold_alloc_uniform(1, B, self.cache.req_to_slot, self.cache.suffix_len, self.cache.cap,
                                        self._slots_buf, st)
            if not fused:
                for layer in range(self.n_layers):
                    self.ctx.cold_append(layer, self._k_buf[layer], self._v_buf[layer], self._slots_buf, B, st)
            for layer in range(self.n_layers):
                if fused:
                    self.ctx.decode_attention_append(layer, self._q_buf[layer], self._k_buf[layer], self._v_buf[layer],
                                                     batch, self.plan, self._o_buf[layer], self._lse_buf[layer], ws,
                                                     ws.numel(), st)
                else:
                    self.ctx.decode_attention(layer, self._q_buf[layer], batch, self.plan, self._o_buf[layer],
                                              self._lse_buf[layer], ws, ws.numel(), st)

        e0.record(s)
        t1 = time.perf_counter()
        issue()
        t_host = time.perf_counter() - t1
        e1.record(s)
        for b in range(B):
            self.cache.seq_len_host[b] += 1
        self.ctx.cold_sync(s)  # host ring position exact before the capture
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):  # on torch's capture stream
            issue()  # recorded, not run
        self._graph, self._graph_key = g, key
        self._cold_dirty = True  # the capture moved the host's copy as if it had run
        return {"dispatch_us": t_disp * 1e6, "host_us": t_host * 1e6, "mode": "capture"}

    def finish_trace(self) -> List[Dict]:
        """Fill in each step's GPU time (synchronises)."""
        torch.cuda.synchronize()
        for rec, (e0, e1) in zip(self.trace, self._events):
            rec["gpu_us"] = e0.elapsed_time(e1) * 1000.0
        self.ctx.sync_status(self.cache.stream())
        return self.trace

    def logical_kv(self, b: int, layer: int):
        """Request b's logical K, V [L_p + len, n_kv, d] (float32), prefix first (keep_logical)."""
        r = self.rows[b]
        pk, pv = self.prefix_kv[r["prefix"]]
        k = np.concatenate([pk[layer]] + r["k"][layer], axis=0)
        v = np.concatenate([pv[layer]] + r["v"][layer], axis=0)
        return k, v


def run(*, steps: int = 64, n_layers: int = 2, prefix_lens=(16384, 4096), start_batch: int = 48,
        p_arrive: float = 0.25, p_complete: float = 0.02, prompt=(64, 512), seed: int = 0,
        max_batch: int = 256, graph: bool = False, headroom: int = 16, fused_append: bool = True) -> Dict:
    """Seeded arrival/completion schedule: each step, with probability p_arrive a request arrives
    (uniform prefix, uniform prompt length in `prompt`), and every active request completes with
    probability p_complete."""
    sched = np.random.default_rng(seed + 1)
    drv = DecodeDriver(prefix_lens=prefix_lens, n_layers=n_layers, max_batch=max_batch,
                       cap=max(prompt) + steps + headroom + 64, seed=seed, graph=graph, headroom=headroom,
                       fused_append=fused_append)
    for i in range(start_batch):
        drv.arrive(int(sched.integers(len(prefix_lens))), int(sched.integers(prompt[0], prompt[1] + 1)))
    for _ in range(steps):
        done = [b for b in range(drv.B) if sched.random() < p_complete]
        for b in sorted(done, reverse=True):
            drv.complete(b)
        while sched.random() < p_arrive and drv.B < max_batch:
            drv.arrive(int(sched.integers(len(prefix_lens))), int(sched.integers(prompt[0], prompt[1] + 1)))
        drv.step()
    trace = drv.finish_trace()
    n_groups = sum(len(t["groups"]) for t in trace)
    n_dense = sum(1 for t in trace for g in t["groups"] if g["backend"] == "dense")
    gpu = [t["gpu_us"] for t in trace]
    disp = [t["dispatch_us"] for t in trace]
    host = [t["host_us"] for t in trace]
    out = {"steps": steps, "layers": n_layers, "graph": graph, "B_min": min(t["B"] for t in trace),
           "B_max": max(t["B"] for t in trace), "dense_fraction": n_dense / max(1, n_groups),
           "gpu_us_per_step_median": statistics.median(gpu),
           "host_us_per_step_median": statistics.median(host),
           "host_share_of_step": statistics.median(h / g for h, g in zip(host, gpu)),
           "dispatch_us_median": statistics.median(disp),
           "dispatch_share_of_step": statistics.median(d / g for d, g in zip(disp, gpu))}
    modes = {}
    for t in trace:
        modes.setdefault(t["mode"], []).append(t["host_us"])
    out["steps_by_mode"] = {m: len(v) for m, v in modes.items()}
    out["host_us_median_by_mode"] = {m: statistics.median(v) for m, v in modes.items()}
    out["trace"] = trace
    return out


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--layers", type=int, default=2)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--trace", action="store_true", help="print every step")
    ap.add_argument("--graph", action="store_true", help="replay each step from a CUDA graph")
    ap.add_argument("--headroom", type=int, default=16, help="tokens a graph's plan allows per request")
    ap.add_argument("--p-arrive", type=float, default=0.25, help="chance of an arrival per step")
    ap.add_argument("--p-complete", type=float, default=0.02, help="chance per request of completing per step")
    ap.add_argument("--no-fused-append", action="store_true", help="append new K/V with launches of their own")
    a = ap.parse_args(argv)
    res = run(steps=a.steps, n_layers=a.layers, seed=a.seed, graph=a.graph, headroom=a.headroom,
              p_arrive=a.p_arrive, p_complete=a.p_complete, fused_append=not a.no_fused_append)
    trace = res.pop("trace")
    if a.trace:
        for i, t in enumerate(trace):
            print(json.dumps({"step": i, **t}))
    print(json.dumps(res))
    return 0


if __name__ == "__main__":
    sys.exit(main())

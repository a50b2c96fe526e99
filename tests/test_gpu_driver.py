"""Multi-step decode with arrivals and completions between steps ("3 GraniKV": the dispatcher
decides per realized batch; "B.4 Per-Step Dispatch Trace"): after several steps of churn the
library's attention for every active request equals the oracle's, computed from the host copies
of the request's logical K/V (its prefix, prompt and decoded tokens), not from the pools."""

import numpy as np
import pytest

from oracle import attention as OA

pytestmark = pytest.mark.gpu


def _assert_batch_close(o, lse, o_ref, lse_ref, what):
    """The parity bounds of every decode test: o max-abs <= 1e-2, mean-abs <= 1e-3 and relative
    L2 error <= 1e-2 (near-uniform softmax rows make |o| small, where the max-abs bound alone
    says little); lse max-abs <= 1e-3."""
    err = np.abs(o - o_ref)
    rel = np.linalg.norm(o - o_ref) / max(np.linalg.norm(o_ref), 1e-30)
    info = f"{what}: max {err.max():.3e} mean {err.mean():.3e} rel {rel:.3e}"
    assert err.max() <= 1e-2 and err.mean() <= 1e-3 and rel <= 1e-2, info
    assert np.abs(lse - lse_ref).max() <= 1e-3, info


def test_driver_churn_matches_oracle(cuda_ok):
    from shared_prefix_kv_decode_gb300.decode_driver import DecodeDriver

    n_q, n_kv, d = 32, 8, 128
    drv = DecodeDriver(prefix_lens=[700, 1500], n_layers=1, n_q=n_q, n_kv=n_kv, head_dim=d, max_batch=64,
                       cap=512, n_slots=40000, seed=3, keep_logical=True)
    sched = np.random.default_rng(7)
    for i in range(20):
        drv.arrive(i % 2, int(sched.integers(1, 200)))
    for step in range(12):
        for b in sorted([b for b in range(drv.B) if sched.random() < 0.1], reverse=True):
            drv.complete(b)
        for _ in range(int(sched.integers(0, 3))):
            drv.arrive(int(sched.integers(2)), int(sched.integers(1, 200)))
        drv.step()
    trace = drv.finish_trace()
    assert len(trace) == 12 and all(t["B"] > 0 and 1 <= len(t["groups"]) <= 2 for t in trace)
    assert all(t["gpu_us"] > 0 and t["dispatch_us"] > 0 for t in trace)
    o, lse = drv.last_out
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    q = drv.last_q[0]
    scale = OA.softmax_scale(d)
    o_ref = np.zeros((drv.B, n_q, d))
    lse_ref = np.zeros((drv.B, n_q))
    for b in range(drv.B):
        K, V = drv.logical_kv(b, 0)
        for h in range(n_q):
            j = OA.kv_head(h, n_q, n_kv)
            o_ref[b, h], lse_ref[b, h] = OA.attend(q[b, h].astype(np.float64), K[:, j].astype(np.float64),
                                                   V[:, j].astype(np.float64), scale)
    _assert_batch_close(o[:drv.B], lse[:drv.B], o_ref, lse_ref, "churn, eager")


def test_driver_graph_replay_matches_oracle(cuda_ok):
    """The step captured in a CUDA graph and replayed (slot allocation, K/V scatter and attention
    of both layers), with a plan made for a small headroom so that it is re-captured as
    requests outgrow it and whenever the batch changes; the last layer's attention of every
    active request equals the oracle's."""
    from shared_prefix_kv_decode_gb300.decode_driver import DecodeDriver

    n_q, n_kv, d, layers = 32, 8, 128, 2
    drv = DecodeDriver(prefix_lens=[900, 300], n_layers=layers, n_q=n_q, n_kv=n_kv, head_dim=d, max_batch=64,
                       cap=512, n_slots=40000, seed=4, keep_logical=True, graph=True, headroom=4)
    sched = np.random.default_rng(8)
    for i in range(12):
        drv.arrive(i % 2, int(sched.integers(1, 150)))
    for step in range(18):
        if step in (6, 13):  # churn between quiet stretches
            drv.complete(int(sched.integers(drv.B)))
            drv.arrive(int(sched.integers(2)), int(sched.integers(1, 150)))
        drv.step()
    trace = drv.finish_trace()
    modes = [t["mode"] for t in trace]
    assert modes.count("replay") >= 8 and modes.count("capture") >= 3, modes
    assert all(t["gpu_us"] > 0 for t in trace)
    o, lse = drv.last_out
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    q = drv.last_q[layers - 1]
    scale = OA.softmax_scale(d)
    o_ref = np.zeros((drv.B, n_q, d))
    lse_ref = np.zeros((drv.B, n_q))
    for b in range(drv.B):
        K, V = drv.logical_kv(b, layers - 1)
        for h in range(n_q):
            j = OA.kv_head(h, n_q, n_kv)
            o_ref[b, h], lse_ref[b, h] = OA.attend(q[b, h].astype(np.float64), K[:, j].astype(np.float64),
                                                   V[:, j].astype(np.float64), scale)
    _assert_batch_close(o[:drv.B], lse[:drv.B], o_ref, lse_ref, "churn, graph replay")
    # once synchronised, the ring position the graph moved on the device accounts for every
    # token the active requests hold (completed requests gave theirs back; prefixes are in HOT)
    drv._sync_cold()
    held = sum(r["len"] for r in drv.rows)
    assert held == sum(drv.cache.seq_len_host[:drv.B])
    n_cold = 40000 - drv.cache.n_hot
    assert drv.cache.ctx.cold_free_count() == n_cold - held

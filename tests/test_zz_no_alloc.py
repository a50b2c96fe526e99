"""granikv_decode_attention_static: decode attention for callers that cannot allocate device
memory (a serving engine that already owns almost all GPU memory, a plain C host holding only
pointers), run on the library's built-in workspace array.

Through the C ABI, on two calls in a row, it must give bit for bit what granikv_decode_attention
gives with a caller workspace (and the oracle's result within the parity tolerances), also when
calls of two plans alternate on the one array; a plan that needs more than the built-in 16 MiB
is refused before anything is enqueued.  This file is collected last on purpose.
"""

import ctypes as C

import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu


def _close(a, b, la, lb):
    err = np.abs(a - b)
    rel = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
    assert err.max() <= 1e-2 and err.mean() <= 1e-3 and rel <= 1e-2
    assert np.abs(la - lb).max() <= 1e-3


def _static_call(ctx, plan, batch, q, n_q, stream):
    import torch
    from shared_prefix_kv_decode_gb300 import _binding as gb
    o = torch.full_like(q, float("nan"))
    lse = torch.full((q.shape[0], n_q), float("nan"), dtype=torch.float32, device=q.device)
    st = ctx._lib.granikv_decode_attention_static(ctx.handle, 0, C.c_void_p(q.data_ptr()), C.byref(batch.c),
                                                  plan.handle, C.c_void_p(o.data_ptr()), C.c_void_p(lse.data_ptr()),
                                                  C.c_void_p(stream.cuda_stream))
    assert st == gb.OK, gb.status_string(st)
    ctx.sync_status(stream)
    return o, lse


def test_static_workspace_matches_caller_workspace(cuda_ok):
    """Two calls in a row through the C ABI equal the caller-workspace call bit for bit (the
    kernels and their work split are the same, only the workspace's address differs), and the
    oracle within the parity tolerances."""
    import torch
    from shared_prefix_kv_decode_gb300.workload_io import load_workload
    import oracle.attention as OA

    wl = W.medium_shared(3, q_scale=1.0)
    lw = load_workload(wl)
    ctx = lw.cache.ctx
    stream = lw.cache.stream()
    plan = ctx.dispatch(lw.batch)
    o_ref, lse_ref = lw.cache.decode(0, lw.q, lw.batch, plan)
    ctx.sync_status(stream)
    for call in range(2):
        o, lse = _static_call(ctx, plan, lw.batch, lw.q, wl.spec.n_q, stream)
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref), call
    o_or, lse_or = OA.decode_attention(wl)
    _close(o.float().cpu().numpy(), o_or, lse.cpu().numpy(), lse_or)


def test_static_workspace_alternating_plans(cuda_ok):
    """Plan A, then plan B (another batch, merged by the last producer of each row, so its merge
    tickets live in the shared array), then plan A again: each call re-copies its own work list
    into the one array and equals its caller-workspace call bit for bit."""
    import torch
    from shared_prefix_kv_decode_gb300 import _binding as gb
    from shared_prefix_kv_decode_gb300.workload_io import load_workload

    wl = W.medium_shared(4, q_scale=1.0)
    lw = load_workload(wl)
    cache, ctx = lw.cache, lw.cache.ctx
    stream = cache.stream()
    n_b = 25
    batch_b = gb.Batch(lw.slab_ids[:n_b], cache.seq_len_host[:n_b], cache.req_to_slot, cache.cap)
    q_b = lw.q[:n_b].contiguous()
    plan_a = ctx.dispatch(lw.batch)
    ctx.set_fused_merge(True)
    plan_b = ctx.dispatch(batch_b)
    ctx.set_fused_merge(False)
    ref = {}
    for name, plan, batch, q in (("a", plan_a, lw.batch, lw.q), ("b", plan_b, batch_b, q_b)):
        o, lse = cache.decode(0, q, batch, plan)
        ctx.sync_status(stream)
        ref[name] = (o.clone(), lse.clone())
    for name in ("a", "b", "a", "b"):
        plan, batch, q = (plan_a, lw.batch, lw.q) if name == "a" else (plan_b, batch_b, q_b)
        o, lse = _static_call(ctx, plan, batch, q, wl.spec.n_q, stream)
        assert torch.equal(o, ref[name][0]) and torch.equal(lse, ref[name][1]), name


def test_static_workspace_refuses_oversized_plans(cuda_ok):
    import torch
    from shared_prefix_kv_decode_gb300 import _binding as gb
    from shared_prefix_kv_decode_gb300.cache import GraniKVCache

    B = 2048
    cache = GraniKVCache(n_layers=1, n_q=32, n_kv=8, head_dim=128, dtype=gb.DTYPE_BF16, n_slots=8192,
                         max_batch=B, cap=8)
    k = torch.zeros((1024, 8, 128), dtype=torch.bfloat16, device="cuda")
    sid = cache.admit_prefix(1024, [k], [k])
    batch = cache.batch([sid] * B, [0] * B)
    plan = cache.ctx.dispatch(batch)
    assert cache.ctx.workspace_size(plan) > 16 << 20
    q = torch.zeros((B, 32, 128), dtype=torch.bfloat16, device="cuda")
    o = torch.zeros_like(q)
    lse = torch.zeros((B, 32), dtype=torch.float32, device="cuda")
    with pytest.raises(gb.GranikvError) as e:
        cache.ctx.decode_attention_static(0, q, batch, plan, o, lse, cache.stream())
    assert e.value.status == gb.ERR_STATIC_WORKSPACE_TOO_SMALL
    cache.ctx.sync_status(cache.stream())
    assert not torch.any(o)  # nothing ran

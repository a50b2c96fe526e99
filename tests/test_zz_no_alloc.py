"""granikv_decode_attention_static: decode attention for callers that cannot allocate device
memory (a serving engine that already owns almost all GPU memory, a plain C host holding only
pointers), run on the library's built-in workspace array.

Through the C ABI, on two calls in a row, it must give what granikv_decode_attention gives with
a caller workspace, within the parity tolerances; a plan that needs more than the built-in
16 MiB is refused before anything is enqueued.  This file is collected last on purpose.
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


def test_static_workspace_matches_caller_workspace(cuda_ok):
    import torch
    from shared_prefix_kv_decode_gb300 import _binding as gb
    from shared_prefix_kv_decode_gb300.workload_io import load_workload

    wl = W.medium_shared(3, q_scale=1.0)
    lw = load_workload(wl)
    ctx = lw.cache.ctx
    stream = lw.cache.stream()
    plan = ctx.dispatch(lw.batch)
    o_ref, lse_ref = lw.cache.decode(0, lw.q, lw.batch, plan)
    ctx.sync_status(stream)
    o_ref = o_ref.float().cpu().numpy()
    lse_ref = lse_ref.cpu().numpy()
    for call in range(2):
        o = torch.full_like(lw.q, float("nan"))
        lse = torch.full((wl.spec.B, wl.spec.n_q), float("nan"), dtype=torch.float32, device=lw.q.device)
        st = ctx._lib.granikv_decode_attention_static(ctx.handle, 0, C.c_void_p(lw.q.data_ptr()),
                                                      C.byref(lw.batch.c), plan.handle,
                                                      C.c_void_p(o.data_ptr()), C.c_void_p(lse.data_ptr()),
                                                      C.c_void_p(stream.cuda_stream))
        assert st == gb.OK, gb.status_string(st)
        ctx.sync_status(stream)
        _close(o.float().cpu().numpy(), o_ref, lse.cpu().numpy(), lse_ref)


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

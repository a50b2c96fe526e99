"""The failure path of the bounded waits, driven from the host without a GPU fault: the test
hook makes one suffix token-CTA withhold the copies of its first tile, so its consumers' wait on
that tile's barrier runs out.  The call must come back with GRANIKV_ERR_DEVICE_CHECK after about
the wait limit (2 s), and the next call on the same context must be correct."""

import time

import numpy as np
import pytest

import oracle.attention as OA
import workloads as W

pytestmark = pytest.mark.gpu


def test_stalled_wait_is_reported_and_the_context_survives(cuda_ok):
    from shared_prefix_kv_decode_gb300 import _binding as gb
    from shared_prefix_kv_decode_gb300.workload_io import load_workload

    wl = W.small_mixed(0, dtype="bf16", q_scale=1.0)
    lw = load_workload(wl, device=0)
    ctx = lw.cache.ctx
    ctx.force_backend(gb.BACKEND_DENSE)
    o_ref, lse_ref = OA.decode_attention(wl)

    def check(o, lse):
        o = o.float().cpu().numpy()
        lse = lse.cpu().numpy()
        assert np.abs(o - o_ref).max() <= 1e-2 and np.abs(lse - lse_ref).max() <= 1e-3

    o, lse = lw.cache.decode(0, lw.q, lw.batch)
    ctx.sync_status(lw.cache.stream())
    check(o, lse)

    ctx.inject_stall(True)
    t0 = time.perf_counter()
    lw.cache.decode(0, lw.q, lw.batch)
    with pytest.raises(gb.DeviceCheckFailed):
        ctx.sync_status(lw.cache.stream())
    waited = time.perf_counter() - t0
    assert 1.5 <= waited <= 30.0, waited  # the 2 s wait limit ran out, once

    o, lse = lw.cache.decode(0, lw.q, lw.batch)
    ctx.sync_status(lw.cache.stream())
    check(o, lse)

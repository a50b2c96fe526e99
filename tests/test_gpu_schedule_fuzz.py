"""GPU parity over seeded random batches, to exercise the dispatcher's scheduling choices:
one grid or kernels one after another, the dense CTAs' L2 read-ahead and their suffix runs,
fixed-length dense pieces with remainders launched last (one prefix length), several prefixes
of one or of different lengths, requests without a HOT prefix, suffix-only and prefix-only
requests.  Each case checks sampled requests against the fp64 oracle (the same tolerances as
the other parity tests) and repeats bit for bit."""

import math

import numpy as np
import pytest

import oracle.attention as OA
import workloads as W

pytestmark = pytest.mark.gpu


def _case(seed: int) -> W.Workload:
    rng = np.random.default_rng(1000 + seed)
    n_q, n_kv = [(32, 8), (40, 8), (16, 8), (64, 8)][seed % 4]
    n_prefix = int(rng.integers(1, 4))
    if seed % 3 == 0:  # prefixes of one length: the serial schedule's remainder pieces
        prefix_lens = [int(rng.integers(256, 20000))] * n_prefix
    else:
        prefix_lens = [int(x) for x in rng.integers(128, 20000, size=n_prefix)]
    B = int(rng.integers(1, 220))
    # mostly requests on a prefix; some with none (a COLD-only request needs a suffix)
    req_prefix = [int(x) if rng.random() > 0.05 else -1 for x in rng.integers(0, n_prefix, size=B)]
    if rng.random() < 0.5:
        suffix = np.clip(rng.lognormal(math.log(300), 1.0, size=B), 0, 2048)
    else:
        suffix = rng.integers(0, 1100, size=B)
    suffix_lens = [int(s) for s in suffix]
    for b in range(B):
        if req_prefix[b] < 0 and suffix_lens[b] == 0:
            suffix_lens[b] = 1
    hot = sum(prefix_lens)
    cold = sum(suffix_lens)
    n_slots = max(int(math.ceil(hot / 0.2)), int(math.ceil(cold / 0.8))) + 4096
    spec = W.WorkloadSpec(
        name=f"fuzz{seed}", dtype="bf16", n_q=n_q, n_kv=n_kv, d=128, prefix_lens=prefix_lens,
        req_prefix=req_prefix, suffix_lens=suffix_lens, q_scale=1.0, n_slots=n_slots,
        schedule_max_chunk=int(rng.choice([1, 16, 64, 512])))
    return W.Workload(spec, seed)


@pytest.mark.parametrize("seed", list(range(12)))
def test_random_batches_match_the_oracle(cuda_ok, seed):
    from shared_prefix_kv_decode_gb300 import _binding as gb
    from shared_prefix_kv_decode_gb300.workload_io import load_workload
    from test_gpu_parity import assert_close

    wl = _case(seed)
    lw = load_workload(wl)
    ctx = lw.cache.ctx
    if seed % 5 == 4:
        ctx.set_concurrency(False, 0.0)
    ctx.force_backend(gb.BACKEND_AUTO)
    plan = ctx.dispatch(lw.batch, ctx.plan())
    o, lse = lw.cache.decode(0, lw.q, lw.batch, plan)
    o2, lse2 = lw.cache.decode(0, lw.q, lw.batch, plan)
    ctx.sync_status(lw.cache.stream())
    import torch
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    B = wl.spec.B
    rng = np.random.default_rng(seed)
    sample = sorted({0, B - 1, *[int(x) for x in rng.integers(0, B, size=3)]})
    o_ref, lse_ref = OA.decode_attention(wl, requests=sample)
    what = (f"seed {seed}: n_q {wl.spec.n_q}, prefixes {wl.spec.prefix_lens}, B {B}, "
            f"schedule {plan.schedule()}, runs {plan.suffix_runs()}, read-ahead {plan.dense_l2_ahead()}")
    assert_close(o[sample], lse[sample], o_ref, lse_ref, "bf16", what)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))


def _case_f32(seed: int) -> W.Workload:
    rng = np.random.default_rng(2000 + seed)
    d = [32, 64, 96, 128, 160, 256][seed % 6]
    n_kv = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.integers(1, 9))
    n_prefix = int(rng.integers(1, 3))
    prefix_lens = [int(x) for x in rng.integers(16, 3000, size=n_prefix)]
    B = int(rng.integers(1, 90))
    req_prefix = [int(x) if rng.random() > 0.1 else -1 for x in rng.integers(0, n_prefix, size=B)]
    suffix_lens = [int(x) for x in rng.integers(0, 300, size=B)]
    for b in range(B):
        if req_prefix[b] < 0 and suffix_lens[b] == 0:
            suffix_lens[b] = 1
    n_slots = max(int(math.ceil(sum(prefix_lens) / 0.2)), int(math.ceil(sum(suffix_lens) / 0.8))) + 2048
    spec = W.WorkloadSpec(
        name=f"fuzz_f32_{seed}", dtype="f32", n_q=n_kv * g, n_kv=n_kv, d=d, prefix_lens=prefix_lens,
        req_prefix=req_prefix, suffix_lens=suffix_lens, q_scale=1.0, n_slots=n_slots,
        schedule_max_chunk=int(rng.choice([1, 16, 64])))
    return W.Workload(spec, seed)


@pytest.mark.parametrize("seed", list(range(6)))
def test_random_fp32_batches_match_the_oracle(cuda_ok, seed):
    """fp32 pools of head sizes 32-256, 1-8 KV heads, GQA groups 1-8, both backends forced and
    dispatched: the tf32 split-precision dense kernel (head sizes up to 128) and the CUDA-core
    kernels hold the fp32 tolerance (1e-5) on sampled requests."""
    from shared_prefix_kv_decode_gb300 import _binding as gb
    from shared_prefix_kv_decode_gb300.workload_io import load_workload
    from test_gpu_parity import assert_close

    wl = _case_f32(seed)
    lw = load_workload(wl)
    ctx = lw.cache.ctx
    B = wl.spec.B
    rng = np.random.default_rng(seed)
    sample = sorted({0, B - 1, *[int(x) for x in rng.integers(0, B, size=3)]})
    o_ref, lse_ref = OA.decode_attention(wl, requests=sample)
    for name, backend in (("auto", gb.BACKEND_AUTO), ("dense", gb.BACKEND_DENSE), ("cascade", gb.BACKEND_CASCADE)):
        ctx.force_backend(backend)
        o, lse = lw.cache.decode(0, lw.q, lw.batch)
        ctx.sync_status(lw.cache.stream())
        o = o.float().cpu().numpy().astype(np.float64)
        lse = lse.cpu().numpy().astype(np.float64)
        what = f"seed {seed} {name}: d {wl.spec.d}, n_kv {wl.spec.n_kv}, g {wl.spec.g}, B {B}, prefixes {wl.spec.prefix_lens}"
        assert_close(o[sample], lse[sample], o_ref, lse_ref, "f32", what)

"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Tolerances, for bf16 inputs with fp32 accumulation: o max-abs <= 1e-2, mean-abs <= 1e-3,
lse max-abs <= 1e-3, plus relative L2 error <= 1e-2 (the near-uniform softmax of the Llama
shape makes |o| ~ 0.01, where an absolute bound alone says little).  fp32 inputs: every path
within 1e-5, the tf32 tensor-core dense path included (it runs each product in split precision,
hi and lo tf32 parts, so its results are fp32-accurate).
Indices (COLD token tables) must match the oracle's ring restatement bit for bit.
"""

import math

import numpy as np
import pytest

import oracle.allocators as AL
import oracle.attention as OA
import workloads as W

pytestmark = pytest.mark.gpu

BACKENDS = ["auto", "dense", "cascade"]


def _gb():
    from shared_prefix_kv_decode_gb300 import _binding as gb
    return gb


def _load(wl, **kw):
    from shared_prefix_kv_decode_gb300.workload_io import load_workload
    return load_workload(wl, **kw)


def _run(lw, backend="auto", requests=None):
    import torch
    gb = _gb()
    ctx = lw.cache.ctx
    ctx.force_backend({"auto": gb.BACKEND_AUTO, "dense": gb.BACKEND_DENSE,
                       "cascade": gb.BACKEND_CASCADE}[backend])
    o, lse = lw.cache.decode(0, lw.q, lw.batch)
    ctx.sync_status(lw.cache.stream())
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    return o, lse


def assert_close(o, lse, o_ref, lse_ref, dtype, what="", dense=False, vmax=None):
    """vmax: for stress inputs far more peaked than the configured workloads, the max-abs bound
    becomes the one bf16 arithmetic guarantees: P and o are each rounded once to bf16 (unit
    roundoff 2^-8), so |o - o_ref| <= 2^-8 (|o_ref| + max|v|)."""
    err = np.abs(o - o_ref)
    lerr = np.abs(lse - lse_ref)
    rel = np.linalg.norm(o - o_ref) / max(np.linalg.norm(o_ref), 1e-30)
    info = f"{what}: max {err.max():.3e} mean {err.mean():.3e} lse {lerr.max():.3e} rel {rel:.3e}"
    if dtype == "f32" and not dense:
        assert err.max() <= 1e-5 and lerr.max() <= 1e-5, info
    else:
        max_abs = 1e-2 if vmax is None else max(1e-2, 2.0 ** -8 * (np.abs(o_ref).max() + vmax))
        assert err.max() <= max_abs, info
        assert err.mean() <= 1e-3, info
        assert lerr.max() <= 1e-3, info
        assert rel <= 1e-2, info


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
@pytest.mark.parametrize("backend", BACKENDS)
def test_tiny_fp32(cuda_ok, seed, backend):
    wl = W.tiny_fp32(seed)
    lw = _load(wl)
    o, lse = _run(lw, backend)
    o_ref, lse_ref = OA.decode_attention(wl)
    assert_close(o, lse, o_ref, lse_ref, "f32", f"tiny seed {seed} {backend}")


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("backend", BACKENDS)
@pytest.mark.parametrize("q_scale", [1.0 / math.sqrt(128.0), 1.0])
def test_small_mixed_bf16(cuda_ok, seed, backend, q_scale):
    """Ragged prefixes (1000, 333), a prefix that fell back to COLD, a prefix-only request, a
    prefix-less request, ragged suffixes; near-uniform and peaked queries."""
    wl = W.small_mixed(seed, dtype="bf16", q_scale=q_scale)
    lw = _load(wl)
    o, lse = _run(lw, backend)
    o_ref, lse_ref = OA.decode_attention(wl)
    assert_close(o, lse, o_ref, lse_ref, "bf16", f"small_mixed seed {seed} {backend} q {q_scale}")


@pytest.mark.parametrize("backend", BACKENDS)
def test_small_mixed_fp32(cuda_ok, backend):
    wl = W.small_mixed(5, dtype="f32", n_q=8, n_kv=2, d=64, q_scale=1.0)
    lw = _load(wl)
    o, lse = _run(lw, backend)
    o_ref, lse_ref = OA.decode_attention(wl)
    assert_close(o, lse, o_ref, lse_ref, "f32", f"small_mixed fp32 {backend}")


@pytest.mark.parametrize("backend", BACKENDS)
@pytest.mark.parametrize("q_scale", [1.0 / math.sqrt(128.0), 1.0, 3.0])
def test_medium_shared_prefix(cuda_ok, backend, q_scale):
    """280 query rows per KV head (three 128-row blocks, the last partial) over a 3000-token
    prefix (several pieces, ragged last tile); q_scale 3 makes the running max jump often."""
    wl = W.medium_shared(1, q_scale=q_scale)
    lw = _load(wl)
    o, lse = _run(lw, backend)
    o_ref, lse_ref = OA.decode_attention(wl)
    vmax = None
    if q_scale > 1.0:  # stress: far more peaked than any configured workload
        vmax = max(np.abs(wl.prefix_v(0)).max(), max(np.abs(wl.suffix_v(b)).max() for b in range(wl.spec.B)))
    assert_close(o, lse, o_ref, lse_ref, "bf16", f"medium {backend} q {q_scale}", vmax=vmax)


@pytest.mark.parametrize("backend", BACKENDS)
def test_needles_locate_the_right_token(cuda_ok, backend):
    """Planted keys in the HOT prefix, in a COLD suffix and in a COLD-resident prefix: the
    output must be the planted token's value, so any gather or slot error is gross."""
    needles = [(0, 17, 3, 30.0), (1, 1005, 0, 30.0), (4, 250, 7, 30.0), (6, 100, 5, 30.0),
               (8, 199, 2, 30.0), (3, 999, 6, 30.0)]
    wl = W.small_mixed(7, dtype="bf16", q_scale=1.0, needles=needles)
    lw = _load(wl)
    o, lse = _run(lw, backend)
    o_ref, lse_ref = OA.decode_attention(wl)
    assert_close(o, lse, o_ref, lse_ref, "bf16", f"needles {backend}")
    for (b, pos, j, _) in needles:
        K, V = OA.logical_kv(wl, b)
        for h in range(j * wl.spec.g, (j + 1) * wl.spec.g):
            assert np.max(np.abs(o[b, h] - V[pos, j])) <= 0.06


def test_cold_tables_match_oracle_ring_bit_exact(cuda_ok):
    wl = W.small_mixed(3, dtype="bf16")
    lw = _load(wl)
    ring = AL.ColdRing(wl.cold_order)
    tables = [[] for _ in range(wl.spec.B)]
    for r in wl.append_schedule:
        ring.alloc([int(x) for x in r], tables)
    got = lw.cache.req_to_slot.cpu().numpy()
    lens = lw.cache.suffix_len.cpu().numpy()
    for b in range(wl.spec.B):
        assert lens[b] == len(tables[b]) == wl.cold_len(b)
        assert list(got[b, :lens[b]]) == tables[b]
    assert lw.cache.ctx.cold_free_count() == ring.n_free


def test_cold_pool_contents_bit_exact(cuda_ok):
    """Every appended token sits in its slot byte for byte, in every layer."""
    import torch
    wl = W.small_mixed(4, dtype="bf16")
    lw = _load(wl, n_layers=2)
    table = lw.cache.req_to_slot.cpu().numpy()
    for layer in range(2):
        kp = lw.cache.k_pools[layer].float().cpu().numpy()
        vp = lw.cache.v_pools[layer].float().cpu().numpy()
        for b in range(wl.spec.B):
            L = wl.cold_len(b)
            assert np.array_equal(kp[table[b, :L]], wl.cold_k(b))
            assert np.array_equal(vp[table[b, :L]], wl.cold_v(b))
        for i, L in enumerate(wl.spec.prefix_lens):
            if not wl.spec.prefix_in_hot[i]:
                continue
            sid = lw.slab_ids[wl.spec.req_prefix.index(i)]
            off, ln = lw.cache.ctx.hot_info(sid)
            assert ln == L
            assert np.array_equal(kp[off:off + L], wl.prefix_k(i))
            assert np.array_equal(vp[off:off + L], wl.prefix_v(i))


@pytest.mark.parametrize("backend", BACKENDS)
def test_cold_slot_permutation_invariance(cuda_ok, backend):
    """Another COLD slot order leaves o and lse unchanged, bit for bit (the kernels' work split
    depends only on lengths, so the arithmetic is the same)."""
    wl1 = W.small_mixed(6, dtype="bf16", q_scale=1.0)
    wl2 = W.small_mixed(6, dtype="bf16", q_scale=1.0)
    rng = np.random.default_rng(99)
    s = wl2.spec
    wl2._cache["cold"] = (s.n_hot + rng.permutation(s.n_slots - s.n_hot)).astype(np.int32)
    o1, l1 = _run(_load(wl1), backend)
    o2, l2 = _run(_load(wl2), backend)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("shape", ["bf16_d128", "f32_d64"])
def test_backends_agree(cuda_ok, shape):
    """Forced dense and forced cascade give the same attention, and are different kernels: bf16
    / head_dim 128 runs the tcgen05 dense kernel against the bandwidth cascade, fp32 the tf32
    tcgen05 dense kernel against the CUDA-core cascade (their outputs differ in the last bits,
    so they are not one kernel run twice).  bf16: within the bf16 bounds of each other; fp32:
    within 2e-5 (each is within 1e-5 of the oracle)."""
    if shape == "f32_d64":
        wl = W.small_mixed(8, dtype="f32", n_q=8, n_kv=2, d=64, q_scale=1.0)
    else:
        wl = W.small_mixed(8, dtype="bf16", q_scale=1.0)
    lw = _load(wl)
    od, ld = _run(lw, "dense")
    oc, lc = _run(lw, "cascade")
    tol_o, tol_l = (2e-5, 2e-5) if shape == "f32_d64" else (1e-2, 1e-3)
    assert np.max(np.abs(od - oc)) <= tol_o and np.max(np.abs(ld - lc)) <= tol_l
    assert not np.array_equal(od, oc)


@pytest.mark.parametrize("d", [32, 64, 96, 128])
@pytest.mark.parametrize("q_scale", [1.0 / 8.0, 1.0])
def test_fp32_dense_tensor_core_head_dims(cuda_ok, d, q_scale):
    """The tf32 dense kernel at every head size it serves (32, 64, 96, 128: one to four 32-wide
    column blocks of the swizzled operands), ragged prefixes (1000 and 333 tokens: ragged last
    32-token tiles) and a peaked query scale, against the oracle within the fp32 bounds."""
    wl = W.small_mixed(6, dtype="f32", n_q=8, n_kv=2, d=d, q_scale=q_scale)
    lw = _load(wl)
    o, lse = _run(lw, "dense")
    o_ref, lse_ref = OA.decode_attention(wl)
    assert_close(o, lse, o_ref, lse_ref, "f32", f"fp32 dense d {d} q {q_scale}")


def test_fp32_dense_several_row_blocks(cuda_ok):
    """fp32, 48 requests of one ragged prefix (g = 4: 192 rows per KV head, two 128-row blocks,
    the second partial) over several L_p pieces: the tf32 dense kernel against the oracle, and
    the CUDA-core cascade backend on the same batch within the fp32 bounds."""
    from workloads.synth import Workload, WorkloadSpec
    rng = np.random.default_rng(11)
    spec = WorkloadSpec(name="fp32_rows", dtype="f32", n_q=8, n_kv=2, d=64, prefix_lens=[1500],
                        req_prefix=[0] * 48, suffix_lens=[int(x) for x in rng.integers(1, 80, size=48)],
                        q_scale=0.5, n_slots=8192, prefix_in_hot=[True], needles=[], schedule_max_chunk=32)
    wl = Workload(spec, 11)
    lw = _load(wl)
    o_ref, lse_ref = OA.decode_attention(wl)
    o, lse = _run(lw, "dense")
    assert_close(o, lse, o_ref, lse_ref, "f32", "fp32 dense 192 rows")
    o, lse = _run(lw, "cascade")
    assert_close(o, lse, o_ref, lse_ref, "f32", "fp32 cascade 192 rows")


@pytest.mark.parametrize("backend", ["dense", "cascade"])
@pytest.mark.parametrize("setting", [(False, 0.5, False), (True, 0.3, False), (True, 1.0, False),
                                     (True, 0.0, False), (False, 0.5, True), (True, 0.3, True),
                                     (True, 0.5, True), (True, 1.0, True), (True, 0.0, True)])
def test_concurrency_and_merge_settings(cuda_ok, backend, setting):
    """The suffix kernel on its own stream next to the prefix kernel (several SM shares, 0 for
    the automatic one) or serial, with the merge kernel or the last-producer merge: every
    setting matches the oracle
    and repeats bit for bit (records are merged in record order, whoever merges them)."""
    wl = W.medium_shared(2, q_scale=1.0)
    lw = _load(wl)
    on, share, fused = setting
    lw.cache.ctx.set_concurrency(on, share)
    lw.cache.ctx.set_fused_merge(fused)
    o, lse = _run(lw, backend)
    o2, lse2 = _run(lw, backend)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    o_ref, lse_ref = OA.decode_attention(wl)
    assert_close(o, lse, o_ref, lse_ref, "bf16", f"concurrency {setting} {backend}")


@pytest.mark.parametrize("serial", [False, True])
def test_dense_l2_read_ahead_leaves_results_unchanged(cuda_ok, serial):
    """The dense kernel's L2 read-ahead only asks for tiles earlier: on the Llama-shape
    workload (16K prefix, 64 requests) every setting gives bit-identical o and lse within a
    schedule (one grid, or the kernels one after another), and they match the oracle."""
    wl = W.llama8b_single_prefix_16k(0)
    lw = _load(wl)
    ctx = lw.cache.ctx
    ctx.set_concurrency(not serial, 0.0)
    got = {}
    for tiles in (0, 2, 7, -1):
        ctx.set_dense_l2_ahead(tiles)
        got[tiles] = _run(lw, "dense")
    ctx.set_dense_l2_ahead(-1)
    for tiles in (2, 7, -1):
        assert np.array_equal(got[tiles][0], got[0][0]) and np.array_equal(got[tiles][1], got[0][1]), tiles
    reqs = [0, 21, 42, 63]
    o_ref, lse_ref = OA.decode_attention(wl, requests=reqs)
    assert_close(got[2][0][reqs], got[2][1][reqs], o_ref, lse_ref, "bf16", f"read-ahead, serial={serial}")


def test_dense_ctas_suffix_runs_match_the_oracle(cuda_ok):
    """Qwen-2.5 shape at full size (16K prefix, B = 128): in the one grid the dense CTAs also
    take suffix runs after their prefix pieces.  Every request with a segment in one of those
    runs is checked against the oracle, and the whole batch repeats bit for bit."""
    import struct
    wl = W.qwen_tp1_16k(0)
    lw = _load(wl)
    ctx = lw.cache.ctx
    ctx.force_backend(_gb().BACKEND_AUTO)
    plan = ctx.dispatch(lw.batch, ctx.plan())
    runs = plan.suffix_runs()
    assert plan.schedule()["concurrent"] and runs["tail_runs"] == plan.schedule()["prefix_ctas"]
    # the suffix items follow the prefix items in the plan image; the run offsets follow them
    B, n_scta = wl.spec.B, runs["runs"]
    img = plan.image()
    a16 = lambda x: (x + 15) // 16 * 16
    off_s = a16(a16(a16(64 + 4 * B) + 16 * B) + 16 * plan.schedule()["prefix_ctas"])
    cb = None
    for n in range(n_scta, (len(img) - off_s) // 16 + 1):
        c = struct.unpack_from("<%di" % (n_scta + 1), img, off_s + 16 * n)
        if c[0] == 0 and c[-1] == n and all(c[i] <= c[i + 1] for i in range(n_scta)):
            cb = c
            break
    assert cb is not None
    first_tail = cb[n_scta - runs["tail_runs"]]
    tail_reqs = sorted({struct.unpack_from("<4i", img, off_s + 16 * i)[0] for i in range(first_tail, cb[-1])})
    assert tail_reqs
    o, lse = lw.cache.decode(0, lw.q, lw.batch, plan)
    o2, lse2 = lw.cache.decode(0, lw.q, lw.batch, plan)
    ctx.sync_status(lw.cache.stream())
    assert torch_equal(o, o2) and torch_equal(lse, lse2)
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    sample = tail_reqs[:: max(1, len(tail_reqs) // 6)][:6]
    o_ref, lse_ref = OA.decode_attention(wl, requests=sample)
    assert_close(o[sample], lse[sample], o_ref, lse_ref, "bf16", f"qwen tail runs {sample}")


def torch_equal(a, b):
    import torch
    return bool(torch.equal(a, b))


def test_run_to_run_deterministic(cuda_ok):
    wl = W.small_mixed(9, dtype="bf16", q_scale=1.0)
    lw = _load(wl)
    for backend in BACKENDS:
        a = _run(lw, backend)
        b = _run(lw, backend)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_device_check_reports_bad_slot_and_context_survives(cuda_ok):
    """A token table entry outside the COLD range is skipped by the kernel's own bounds check
    and reported as a device check failure; the context keeps working afterwards."""
    gb = _gb()
    wl = W.small_mixed(10, dtype="bf16")
    lw = _load(wl)
    good = lw.cache.req_to_slot.clone()
    lw.cache.req_to_slot[4, 3] = 0  # slot 0 is HOT, not COLD
    with pytest.raises(gb.DeviceCheckFailed):
        _run(lw, "cascade")
    lw.cache.req_to_slot.copy_(good)
    o, lse = _run(lw, "cascade")
    o_ref, lse_ref = OA.decode_attention(wl)
    assert_close(o, lse, o_ref, lse_ref, "bf16", "after device check")


def test_cold_exhaustion_is_all_or_nothing(cuda_ok):
    import torch
    gb = _gb()
    from shared_prefix_kv_decode_gb300.cache import GraniKVCache
    cache = GraniKVCache(n_layers=1, n_q=8, n_kv=2, head_dim=64, dtype=gb.DTYPE_F32, n_slots=100,
                         max_batch=3, cap=64)
    free0 = cache.ctx.cold_free_count()
    assert free0 == 80
    k = torch.zeros((70, 2, 64), device="cuda")
    cache.append([30, 0, 40], [k], [k])
    assert cache.ctx.cold_free_count() == 10
    with pytest.raises(gb.NoColdSpace):
        cache.append([5, 5, 5], [k[:15]], [k[:15]])
    assert cache.ctx.cold_free_count() == 10
    assert cache.suffix_len.cpu().tolist() == [30, 0, 40]


def test_cold_free_returns_slots_fifo(cuda_ok):
    import torch
    gb = _gb()
    from shared_prefix_kv_decode_gb300.cache import GraniKVCache
    order = list(range(20, 100))[::-1]
    cache = GraniKVCache(n_layers=1, n_q=8, n_kv=2, head_dim=64, dtype=gb.DTYPE_F32, n_slots=100,
                         max_batch=2, cap=128, cold_init_order=order)
    ring = AL.ColdRing(order)
    tables = [[], []]
    k = torch.zeros((80, 2, 64), device="cuda")
    cache.append([50, 30], [k], [k])
    ring.alloc([50, 30], tables)
    freed = torch.tensor(tables[0][:20], dtype=torch.int32, device="cuda")
    cache.ctx.cold_free(freed, 20, cache.stream())
    ring.free(tables[0][:20])
    cache.append([0, 15], [k[:15]], [k[:15]])
    ring.alloc([0, 15], tables)
    got = cache.req_to_slot.cpu().numpy()
    assert list(got[1, :45]) == tables[1]
    cache.ctx.sync_status()


def test_cold_alloc_uniform_follows_the_ring(cuda_ok):
    """The graph-safe allocation (ring position kept on the device) takes exactly the slots the
    oracle's FIFO ring gives, mixed with the host-driven allocation and frees; when too few are
    free it pops nothing and reports a device check."""
    import torch
    gb = _gb()
    from shared_prefix_kv_decode_gb300.cache import GraniKVCache
    order = [int(x) for x in np.random.default_rng(3).permutation(np.arange(20, 100))]
    cache = GraniKVCache(n_layers=1, n_q=8, n_kv=2, head_dim=64, dtype=gb.DTYPE_F32, n_slots=100,
                         max_batch=4, cap=64, cold_init_order=order)
    ring = AL.ColdRing(order)
    tables = [[], [], [], []]
    s = cache.stream()
    k = torch.zeros((40, 2, 64), device="cuda")
    slots = torch.zeros((16,), dtype=torch.int32, device="cuda")
    cache.append([3, 0, 5, 1], [k[:9]], [k[:9]])
    ring.alloc([3, 0, 5, 1], tables)
    for n in (1, 2, 1):
        cache.ctx.cold_alloc_uniform(n, 4, cache.req_to_slot, cache.suffix_len, cache.cap, slots, s)
        want = ring.alloc([n] * 4, tables)
        assert slots[:4 * n].cpu().tolist() == want
    cache.ctx.cold_sync(s)
    assert cache.ctx.cold_free_count() == ring.n_free
    # frees after device-side allocations, then both kinds again
    cache.ctx.cold_free(torch.tensor(tables[2][:4], dtype=torch.int32, device="cuda"), 4, s)
    ring.free(tables[2][:4])
    cache.ctx.cold_alloc_uniform(1, 3, cache.req_to_slot, cache.suffix_len, cache.cap, slots, s)
    ring.alloc([1, 1, 1, 0], tables)
    cache.ctx.cold_sync(s)
    cache.append([2, 2, 0, 0], [k[:4]], [k[:4]])
    ring.alloc([2, 2, 0, 0], tables)
    got = cache.req_to_slot.cpu().numpy()
    lens = cache.suffix_len.cpu().tolist()
    for b in range(4):
        assert lens[b] == len(tables[b]) and list(got[b, :lens[b]]) == tables[b], b
    cache.ctx.cold_sync(s)
    assert cache.ctx.cold_free_count() == ring.n_free
    # asking for more than is free: nothing popped, the device check is reported
    free = ring.n_free
    big = free // 4 + 1
    before = cache.req_to_slot.clone(), cache.suffix_len.clone()
    cache.ctx.cold_alloc_uniform(big, 4, cache.req_to_slot, cache.suffix_len, cache.cap, None, s)
    with pytest.raises(gb.DeviceCheckFailed):
        cache.ctx.sync_status(s)
    cache.ctx.cold_sync(s)
    assert cache.ctx.cold_free_count() == free
    assert torch.equal(cache.req_to_slot, before[0]) and torch.equal(cache.suffix_len, before[1])


FULL = {
    "llama8b_single_prefix_16k": (W.llama8b_single_prefix_16k, [0, 17, 40, 63]),
    "hetero_multi_prefix_k8": (W.hetero_multi_prefix_k8, [0, 31, 77, 159]),
    "qwen_tp1_16k": (W.qwen_tp1_16k, [0, 64, 127]),
}


@pytest.mark.parametrize("name", sorted(FULL))
def test_full_size_sampled(cuda_ok, name):
    """Full-size configurations, the same launch configuration the benchmark times, checked on
    sampled requests the oracle computes one by one, for every backend."""
    fn, sample = FULL[name]
    wl = fn(0)
    lw = _load(wl)
    refs = {b: OA.request_attention(wl, b) for b in sample}
    for backend in BACKENDS:
        o, lse = _run(lw, backend)
        for b in sample:
            assert_close(o[b], lse[b], refs[b][0], refs[b][1], "bf16", f"{name} b={b} {backend}")
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))


@pytest.mark.parametrize("backend", BACKENDS)
def test_slab_fills_hot_and_table_fills_cap(cuda_ok, backend):
    """A prefix as long as the whole HOT range (1638 of 8192 slots: the slab ends exactly at the
    HOT/COLD boundary) and a token table filled to its capacity (64 COLD tokens, cap 64), next
    to a short suffix and an empty one."""
    spec = W.WorkloadSpec(name="hot_full", dtype="bf16", n_q=32, n_kv=8, d=128, prefix_lens=[1638],
                          req_prefix=[0, 0, 0], suffix_lens=[64, 5, 0], q_scale=1.0, n_slots=8192)
    wl = W.Workload(spec, 9)
    lw = _load(wl, cap=64)
    off, L = lw.cache.ctx.hot_info(lw.slab_ids[0])
    assert off == 0 and off + L == lw.cache.n_hot
    o, lse = _run(lw, backend)
    o_ref, lse_ref = OA.decode_attention(wl)
    assert_close(o, lse, o_ref, lse_ref, "bf16", f"HOT-filling slab {backend}")


def test_largest_batch(cuda_ok):
    """B = 4096, the default largest batch of a context: two prefixes (384 and 1000 tokens),
    requests alternating between them, 1-8 COLD tokens each.  The dense kernel runs 64 row
    blocks per KV head and group (8192 rows), the merge 131,072 rows, each suffix token-CTA
    dozens of requests.  Every backend, checked on sampled requests the oracle computes
    one by one; every output finite."""
    B = 4096
    rng = np.random.default_rng(4096)
    spec = W.WorkloadSpec(name="largest_batch", dtype="bf16", n_q=32, n_kv=8, d=128, prefix_lens=[384, 1000],
                          req_prefix=[b % 2 for b in range(B)],
                          suffix_lens=[int(x) for x in rng.integers(1, 9, size=B)], q_scale=1.0,
                          n_slots=65536, schedule_max_chunk=8)
    wl = W.Workload(spec, 5)
    lw = _load(wl)
    sample = [0, 1, 2, 1023, 2048, 2049, 3333, 4094, 4095]
    refs = {b: OA.request_attention(wl, b) for b in sample}
    for backend in BACKENDS:
        o, lse = _run(lw, backend)
        for b in sample:
            assert_close(o[b], lse[b], refs[b][0], refs[b][1], "bf16", f"largest batch b={b} {backend}")
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))


@pytest.mark.parametrize("backend", ["dense", "cascade"])
def test_hot_layout_equals_paged_equivalent_layout(cuda_ok, backend):
    """The comparator's batch (one shared prefix, every request with its own suffix) stored with
    the prefix in one HOT slab, or copied at the head of every request's COLD token table (the
    paged-equivalent layout, "B.10"), each matches the oracle on the generator's logical arrays
    ("Ethics Statement": the layer changes layout and kernel choice, not outputs)."""
    import torch
    gb = _gb()
    from shared_prefix_kv_decode_gb300.layout_bench import build
    cache_h, batch_h, q, wl = build(1000, 8, 50, paged=False, seed=3)
    o_ref, lse_ref = OA.decode_attention(wl)
    cache_h.ctx.force_backend({"dense": gb.BACKEND_DENSE, "cascade": gb.BACKEND_CASCADE}[backend])
    o_h, l_h = cache_h.decode(0, q, batch_h)
    cache_h.ctx.sync_status(cache_h.stream())
    assert_close(o_h.float().cpu().numpy().astype(np.float64), l_h.cpu().numpy().astype(np.float64),
                 o_ref, lse_ref, "bf16", f"HOT layout {backend}")
    cache_p, batch_p, q2, _ = build(1000, 8, 50, paged=True, seed=3)
    assert torch.equal(q, q2)
    o_p, l_p = cache_p.decode(0, q2, batch_p)
    cache_p.ctx.sync_status(cache_p.stream())
    assert_close(o_p.float().cpu().numpy().astype(np.float64), l_p.cpu().numpy().astype(np.float64),
                 o_ref, lse_ref, "bf16", "paged-equivalent layout")


SWEEP_CELLS = [(lp, b) for lp in (512, 2048, 32768) for b in (256, 512)]


@pytest.mark.parametrize("L_p,B", SWEEP_CELLS)
def test_dispatch_sweep_large_cells(cuda_ok, L_p, B):
    """Cells of the L_p x B crossover sweep ("B.4 Per-Step Dispatch Trace"; "Limitations": the
    small-L_p / high-B corner) at the batch sizes where the dense kernel runs 8 or 16 row blocks
    per KV head, 256 COLD tokens per request, with each forced backend and the dispatcher's own
    choice.  Sampled requests: the first, middle and last 128-row block of each KV head (32
    requests a block at g = 4), and two planted needles in the last block: one in the shared
    prefix's last tile (KV head 5) and one in a request's own suffix (KV head 2)."""
    g = 4
    needles = [(B - 2, L_p - 3, 5, 30.0), (B - 1, L_p + 100, 2, 30.0)]
    wl = W.dispatch_sweep_cell(L_p, B, seed=L_p + B, needles=needles)
    lw = _load(wl)
    rows = 128 // g
    mid = (B // rows // 2) * rows
    sample = sorted({0, rows - 1, mid, mid + rows - 1, B - rows, B - 3, B - 2, B - 1})
    refs = {b: OA.request_attention(wl, b) for b in sample}
    for backend in BACKENDS:
        o, lse = _run(lw, backend)
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
        for b in sample:
            assert_close(o[b], lse[b], refs[b][0], refs[b][1], "bf16", f"Lp {L_p} B {B} b={b} {backend}")
        for (b, pos, j, _) in needles:
            K, V = OA.logical_kv(wl, b)
            for h in range(j * g, (j + 1) * g):
                assert np.max(np.abs(o[b, h] - V[pos, j])) <= 0.06, (backend, b, h)


def test_full_size_whole_batch_through_the_benchmarked_call(cuda_ok):
    """The call the benchmark times -- granikv_decode_attention_append on the Llama-shape
    workload (16384-token prefix, 64 requests, log-normal suffixes), automatic split, one grid
    -- checked on every request and head against the oracle, whose key sequence for request b is
    the prefix, its suffix, and the step's new token."""
    import torch
    gb = _gb()
    wl = W.llama8b_single_prefix_16k(0)
    lw = _load(wl)
    cache, ctx, spec = lw.cache, lw.cache.ctx, wl.spec
    B, s = spec.B, cache.stream()
    rng = np.random.default_rng(11)
    kn = W.round_to_bf16(rng.standard_normal((B, spec.n_kv, 128), dtype=np.float32))
    vn = W.round_to_bf16(rng.standard_normal((B, spec.n_kv, 128), dtype=np.float32))
    kn_d = torch.from_numpy(kn).cuda().to(torch.bfloat16)
    vn_d = torch.from_numpy(vn).cuda().to(torch.bfloat16)
    slots = torch.empty((B,), dtype=torch.int32, device="cuda")
    ctx.cold_alloc([1] * B, cache.req_to_slot, cache.suffix_len, cache.cap, slots, s)
    batch = gb.Batch(lw.slab_ids, [cache.seq_len_host[b] + 1 for b in range(B)], cache.req_to_slot, cache.cap)
    plan = ctx.dispatch(batch)
    sched = plan.schedule()
    assert sched["concurrent"] and sched["prefix_ctas"] + sched["suffix_ctas"] == 152
    assert plan.dense_l2_ahead() == 2  # the dense CTAs read ahead into L2 in this split
    ws = cache.workspace(plan)
    o = torch.empty((B, spec.n_q, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, spec.n_q), dtype=torch.float32, device="cuda")
    ctx.decode_attention_append(0, lw.q, kn_d, vn_d, batch, plan, o, lse, ws, ws.numel(), s)
    ctx.sync_status(s)
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    scale = OA.softmax_scale(128)
    o_ref = np.zeros_like(o)
    lse_ref = np.zeros_like(lse)
    for b in range(B):
        K, V = OA.logical_kv(wl, b)
        K = np.concatenate([K, kn[b][None].astype(np.float64)])
        V = np.concatenate([V, vn[b][None].astype(np.float64)])
        for h in range(spec.n_q):
            j = OA.kv_head(h, spec.n_q, spec.n_kv)
            o_ref[b, h], lse_ref[b, h] = OA.attend(wl.q[b, h], K[:, j], V[:, j], scale)
    assert_close(o, lse, o_ref, lse_ref, "bf16", "llama8b whole batch, fused append")


@pytest.mark.parametrize("shape", [(32, 16), (8, 8), (64, 8), (16, 2), (64, 2), (160, 1)])
@pytest.mark.parametrize("backend", BACKENDS)
def test_head_shapes(cuda_ok, shape, backend):
    """GQA shapes besides the configurations': more than eight KV heads (two head groups in the
    suffix and streaming cascade kernels), one query head per KV head (g = 1), g = 8, two KV
    heads, g = 32 (the streaming cascade with several warps a KV head; the CUDA-core suffix
    kernel) and g = 160 (past the streaming cascade's 128 query columns: the warp-MMA cascade
    kernel; a request's rows span two 128-row dense blocks); bf16, d = 128, the small mixed batch
    (ragged prefixes, a prefix-only and a prefix-less request)."""
    n_q, n_kv = shape
    wl = W.small_mixed(4, dtype="bf16", n_q=n_q, n_kv=n_kv, q_scale=1.0)
    lw = _load(wl)
    o, lse = _run(lw, backend)
    o_ref, lse_ref = OA.decode_attention(wl)
    assert_close(o, lse, o_ref, lse_ref, "bf16", f"heads {shape} {backend}")


@pytest.mark.parametrize("backend", BACKENDS)
@pytest.mark.parametrize("lens", [(100, 5), (128, 0), (1, 1), (129, 16)])
def test_single_request(cuda_ok, backend, lens):
    """B = 1: a prefix shorter than, equal to and one token past a 128-token tile, with a short
    or empty suffix (and a one-token prefix with a one-token suffix)."""
    L_p, L_s = lens
    spec = W.WorkloadSpec(name="single", dtype="bf16", n_q=32, n_kv=8, d=128, prefix_lens=[L_p],
                          req_prefix=[0], suffix_lens=[L_s], q_scale=1.0, n_slots=4096)
    wl = W.Workload(spec, 11)
    lw = _load(wl)
    o, lse = _run(lw, backend)
    o_ref, lse_ref = OA.decode_attention(wl)
    assert_close(o, lse, o_ref, lse_ref, "bf16", f"single {lens} {backend}")


@pytest.mark.parametrize("backend", ["dense", "cascade"])
def test_fp32_tile_boundaries(cuda_ok, backend):
    """fp32 (d = 64): prefixes of 1, 31, 32, 33 and 65 tokens (around the tf32 dense kernel's
    32-token tiles and the CUDA-core kernel's), groups of 1 to 3 requests, suffixes of 0 to 2
    tokens, within the fp32 bounds."""
    lps = [1, 31, 32, 33, 65]
    req_prefix = [0, 1, 1, 2, 2, 2, 3, 4, 4]
    spec = W.WorkloadSpec(name="fp32_edges", dtype="f32", n_q=8, n_kv=2, d=64, prefix_lens=lps,
                          req_prefix=req_prefix, suffix_lens=[i % 3 for i in range(len(req_prefix))],
                          q_scale=1.0, n_slots=4096)
    wl = W.Workload(spec, 17)
    lw = _load(wl)
    o, lse = _run(lw, backend)
    o_ref, lse_ref = OA.decode_attention(wl)
    assert_close(o, lse, o_ref, lse_ref, "f32", f"fp32 tile edges {backend}")


@pytest.mark.parametrize("shape,prefix_lens,group_sizes", [
    ((32, 8), [5000, 3001, 777, 2500], [1, 2, 4, 5]),
    ((40, 8), [4100, 1500], [3, 4]),
])
@pytest.mark.parametrize("q_scale", [1.0 / math.sqrt(128), 1.0])
def test_cascade_small_row_blocks(cuda_ok, shape, prefix_lens, group_sizes, q_scale):
    """The cascade kernel on groups whose query rows fit one warp (B_g * g <= 16: 4, 8, 16 and
    15 rows), where the eight warps split each tile's tokens and merge their states, next to
    groups of 20 rows in the same launch; prefixes of many tiles with ragged last tiles."""
    n_q, n_kv = shape
    req_prefix = [i for i, n in enumerate(group_sizes) for _ in range(n)]
    rng = np.random.default_rng(sum(prefix_lens) + n_q)
    spec = W.WorkloadSpec(name="cascade_small_blocks", dtype="bf16", n_q=n_q, n_kv=n_kv, d=128,
                          prefix_lens=list(prefix_lens), req_prefix=req_prefix,
                          suffix_lens=[int(x) for x in rng.integers(0, 40, size=len(req_prefix))],
                          q_scale=q_scale, n_slots=65536)
    wl = W.Workload(spec, 21)
    lw = _load(wl)
    o, lse = _run(lw, "cascade")
    assert all(gr["backend"] == _gb().BACKEND_CASCADE for gr in lw.cache.ctx.dispatch(lw.batch).groups())
    o_ref, lse_ref = OA.decode_attention(wl)
    assert_close(o, lse, o_ref, lse_ref, "bf16", f"cascade small blocks {shape} {group_sizes}")


@pytest.mark.parametrize("n_kv", [8, 16])
def test_fused_append_equals_append_then_attention(cuda_ok, n_kv):
    """granikv_decode_attention_append (the step's new K/V read by the suffix kernel and written
    to their slots by it) gives bit for bit the o, lse and pools of granikv_cold_append followed
    by granikv_decode_attention; also with a plan made for a headroom and the live lengths read
    from the device."""
    import torch
    gb = _gb()
    wl = W.small_mixed(2, dtype="bf16", n_q=32, n_kv=n_kv, q_scale=1.0)
    lw = _load(wl)
    cache, ctx, spec = lw.cache, lw.cache.ctx, wl.spec
    B, s = spec.B, lw.cache.stream()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(7)
    kn = torch.randn((B, n_kv, 128), generator=gen, device="cuda").to(torch.bfloat16)
    vn = torch.randn((B, n_kv, 128), generator=gen, device="cuda").to(torch.bfloat16)
    slots = torch.empty((B,), dtype=torch.int32, device="cuda")
    ctx.cold_alloc([1] * B, cache.req_to_slot, cache.suffix_len, cache.cap, slots, s)
    lens = [cache.seq_len_host[b] + 1 for b in range(B)]
    pools0 = cache.k_pools[0].clone(), cache.v_pools[0].clone()
    for headroom, live in ((0, None), (5, cache.suffix_len)):
        batch = gb.Batch(lw.slab_ids, [n + headroom for n in lens], cache.req_to_slot, cache.cap, seq_len_dev=live)
        plan = ctx.dispatch(batch)
        ws = cache.workspace(plan)
        outs = []
        for fused in (True, False):
            cache.k_pools[0].copy_(pools0[0])
            cache.v_pools[0].copy_(pools0[1])
            o = torch.empty((B, spec.n_q, 128), dtype=torch.bfloat16, device="cuda")
            lse = torch.empty((B, spec.n_q), dtype=torch.float32, device="cuda")
            if fused:
                ctx.decode_attention_append(0, lw.q, kn, vn, batch, plan, o, lse, ws, ws.numel(), s)
            else:
                ctx.cold_append(0, kn, vn, slots, B, s)
                ctx.decode_attention(0, lw.q, batch, plan, o, lse, ws, ws.numel(), s)
            ctx.sync_status(s)
            outs.append((o.clone(), lse.clone(), cache.k_pools[0].clone(), cache.v_pools[0].clone()))
        for a, b in zip(outs[0], outs[1]):
            assert torch.equal(a, b), headroom
    # refusals, before anything is launched
    bad = gb.Batch(lw.slab_ids, [0] + lens[1:], cache.req_to_slot, cache.cap)
    if lw.slab_ids[0] >= 0:
        plan = ctx.dispatch(bad)
        with pytest.raises(gb.GranikvError) as ei:
            ctx.decode_attention_append(0, lw.q, kn, vn, bad, plan, o, lse, ws, ws.numel(), s)
        assert ei.value.status == gb.ERR_INVALID
    batch = gb.Batch(lw.slab_ids, lens, cache.req_to_slot, cache.cap)
    plan = ctx.dispatch(batch)
    flat = kn.view(-1)
    with pytest.raises(gb.GranikvError) as ei:
        ctx.decode_attention_append(0, lw.q, flat[1:1 + kn.numel() - 8], vn, batch, plan, o, lse, ws, ws.numel(), s)
    assert ei.value.status == gb.ERR_INVALID


def test_fused_append_generic_path(cuda_ok):
    """fp32 and a head size without a tensor-core kernel: the generic suffix kernel takes the
    newest token from k_new/v_new and writes it to its slot, bit for bit as append + attention."""
    import torch
    gb = _gb()
    wl = W.small_mixed(4, dtype="f32", n_q=8, n_kv=2, d=64)
    lw = _load(wl)
    cache, ctx, spec = lw.cache, lw.cache.ctx, wl.spec
    B, s = spec.B, cache.stream()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(9)
    kn = torch.randn((B, 2, 64), generator=gen, device="cuda")
    vn = torch.randn((B, 2, 64), generator=gen, device="cuda")
    slots = torch.empty((B,), dtype=torch.int32, device="cuda")
    ctx.cold_alloc([1] * B, cache.req_to_slot, cache.suffix_len, cache.cap, slots, s)
    batch = gb.Batch(lw.slab_ids, [cache.seq_len_host[b] + 1 for b in range(B)], cache.req_to_slot, cache.cap)
    plan = ctx.dispatch(batch)
    ws = cache.workspace(plan)
    pools0 = cache.k_pools[0].clone(), cache.v_pools[0].clone()
    outs = []
    for fused in (True, False):
        cache.k_pools[0].copy_(pools0[0])
        cache.v_pools[0].copy_(pools0[1])
        o = torch.empty((B, 8, 64), device="cuda")
        lse = torch.empty((B, 8), device="cuda")
        if fused:
            ctx.decode_attention_append(0, lw.q, kn, vn, batch, plan, o, lse, ws, ws.numel(), s)
        else:
            ctx.cold_append(0, kn, vn, slots, B, s)
            ctx.decode_attention(0, lw.q, batch, plan, o, lse, ws, ws.numel(), s)
        ctx.sync_status(s)
        outs.append((o.clone(), lse.clone(), cache.k_pools[0].clone(), cache.v_pools[0].clone()))
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["llama8b_single_prefix_16k", "qwen_tp1_16k"])
def test_fused_append_full_size(cuda_ok, name):
    """At full size, in the launch configuration the benchmark times (automatic split, one grid),
    one decode step with the fused append equals append + attention bit for bit, and the
    split is the one the benchmark reports."""
    import torch
    gb = _gb()
    wl = FULL[name][0](0)
    lw = _load(wl)
    cache, ctx, spec = lw.cache, lw.cache.ctx, wl.spec
    B, s = spec.B, cache.stream()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(3)
    kn = torch.randn((B, spec.n_kv, 128), generator=gen, device="cuda").to(torch.bfloat16)
    vn = torch.randn((B, spec.n_kv, 128), generator=gen, device="cuda").to(torch.bfloat16)
    slots = torch.empty((B,), dtype=torch.int32, device="cuda")
    ctx.cold_alloc([1] * B, cache.req_to_slot, cache.suffix_len, cache.cap, slots, s)
    batch = gb.Batch(lw.slab_ids, [cache.seq_len_host[b] + 1 for b in range(B)], cache.req_to_slot, cache.cap)
    plan = ctx.dispatch(batch)
    sched = plan.schedule()
    assert sched["concurrent"] and sched["prefix_ctas"] + sched["suffix_ctas"] == 152
    ws = cache.workspace(plan)
    pools0 = cache.k_pools[0].clone(), cache.v_pools[0].clone()
    outs = []
    for fused in (True, False):
        cache.k_pools[0].copy_(pools0[0])
        cache.v_pools[0].copy_(pools0[1])
        o = torch.empty((B, spec.n_q, 128), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((B, spec.n_q), dtype=torch.float32, device="cuda")
        if fused:
            ctx.decode_attention_append(0, lw.q, kn, vn, batch, plan, o, lse, ws, ws.numel(), s)
        else:
            ctx.cold_append(0, kn, vn, slots, B, s)
            ctx.decode_attention(0, lw.q, batch, plan, o, lse, ws, ws.numel(), s)
        ctx.sync_status(s)
        outs.append((o.clone(), lse.clone(), cache.k_pools[0].clone(), cache.v_pools[0].clone()))
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)

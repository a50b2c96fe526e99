"""Causal prefill of a HOT slab on the GPU against the oracle's causal_prefill: every token and
head at small, ragged sizes (including L_p = 1 and lengths that are not multiples of a tile),
sampled tokens at L_p = 16384, several GQA group sizes, the slab placed after another one, and
every pool row outside the slab poisoned with NaN so that a masked key that leaked into a sum
would show.

GraniKV (arXiv:2608.15584): "2 Related Work" (a prefix is prefilled once and then reused) and the
card page (the HOT slab holds the prefix's K_p contiguously)."""

import math

import numpy as np
import pytest

from oracle import attention as OA

pytestmark = pytest.mark.gpu

D = 128


def _run(n_q, n_kv, L_p, q_scale, seed, tokens=None):
    import torch
    from shared_prefix_kv_decode_gb300 import _binding as gb
    from shared_prefix_kv_decode_gb300.cache import GraniKVCache
    rng = np.random.default_rng(seed)
    n_slots = int(math.ceil((L_p + 300) / 0.2)) + 64
    cache = GraniKVCache(n_layers=1, n_q=n_q, n_kv=n_kv, head_dim=D, dtype=gb.DTYPE_BF16, n_slots=n_slots,
                         max_batch=4, cap=16)
    cache.k_pools[0].fill_(float("nan"))
    cache.v_pools[0].fill_(float("nan"))
    cache.ctx.hot_alloc(257)  # the prefix's slab starts at slot 257
    sid, off = cache.ctx.hot_alloc(L_p)
    assert off == 257

    def bf(shape, scale=1.0):
        x = rng.standard_normal(shape, dtype=np.float32) * np.float32(scale)
        return torch.from_numpy(x).to(torch.bfloat16)

    q, k, v = bf((L_p, n_q, D), q_scale), bf((L_p, n_kv, D)), bf((L_p, n_kv, D))
    o, lse = cache.prefill(0, sid, q.cuda(), k.cuda(), v.cuda())
    cache.ctx.sync_status(cache.stream())
    assert torch.equal(cache.k_pools[0][off:off + L_p].cpu(), k)
    assert torch.equal(cache.v_pools[0][off:off + L_p].cpu(), v)
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    toks = list(range(L_p)) if tokens is None else tokens
    o_ref, lse_ref = OA.causal_prefill(q.float().numpy(), k.float().numpy(), v.float().numpy(), tokens=toks)
    err_o = np.abs(o[toks] - o_ref)
    err_l = np.abs(lse[toks] - lse_ref)
    assert np.all(np.isfinite(o[toks])) and np.all(np.isfinite(lse[toks]))
    # o leaves the kernel rounded to bf16 and every softmax weight enters the PV product rounded
    # to bf16, each a relative error of at most 2^-9, so the bound scales with |o|: the decode
    # bound 1e-2 up to |o| = 1 and 1% (about 2.5 bf16 ulps) above it.  Early tokens average a
    # few value rows only, so there |o| reaches 3-4.
    rel = err_o / np.maximum(1.0, np.abs(o_ref))
    assert rel.max() <= 1e-2 and err_o.mean() <= 1e-3, (rel.max(), err_o.max(), err_o.mean())
    assert err_l.max() <= 1e-3, err_l.max()


@pytest.mark.parametrize("L_p", [1, 5, 31, 32, 127, 128, 129, 333, 1000])
def test_prefill_llama_heads(cuda_ok, L_p):
    _run(32, 8, L_p, 1.0 / math.sqrt(128), seed=L_p)


@pytest.mark.parametrize("n_q,n_kv,L_p", [(64, 8, 300), (8, 8, 260), (16, 8, 517), (32, 2, 400),
                                         (40, 8, 611), (24, 8, 300), (56, 8, 129)])
def test_prefill_group_sizes(cuda_ok, n_q, n_kv, L_p):
    _run(n_q, n_kv, L_p, 1.0, seed=n_q + L_p)


def test_prefill_sharp_scores(cuda_ok):
    # q ~ N(0, 1): peaked softmax rows, the running max moves often
    _run(32, 8, 700, 1.0, seed=9)


def test_prefill_full_size_sampled(cuda_ok):
    rng = np.random.default_rng(1)
    toks = sorted(set([0, 1, 31, 32, 127, 128, 4095, 8191, 16383] +
                      [int(x) for x in rng.integers(0, 16384, size=16)]))
    _run(32, 8, 16384, 1.0 / math.sqrt(128), seed=2, tokens=toks)


def test_prefill_qwen_shape_full_size_sampled(cuda_ok):
    # 40/8 heads: g = 5 does not divide the 128-row block, so blocks straddle tokens and tiles
    rng = np.random.default_rng(4)
    toks = sorted(set([0, 1, 25, 26, 127, 128, 8191] + [int(x) for x in rng.integers(0, 8192, size=12)]))
    _run(40, 8, 8192, 1.0 / math.sqrt(128), seed=5, tokens=toks)


def test_prefill_refuses_unsupported(cuda_ok):
    import torch
    from shared_prefix_kv_decode_gb300 import _binding as gb
    from shared_prefix_kv_decode_gb300.cache import GraniKVCache
    cache = GraniKVCache(n_layers=1, n_q=8, n_kv=2, head_dim=64, dtype=gb.DTYPE_F32, n_slots=4096,
                         max_batch=4, cap=16)
    sid, _ = cache.ctx.hot_alloc(100)
    q = torch.zeros((100, 8, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(gb.GranikvError) as ei:
        cache.prefill(0, sid, q)
    assert ei.value.status == gb.ERR_UNSUPPORTED
    with pytest.raises(gb.GranikvError) as ei:
        cache.prefill(0, sid + 5, q)
    assert ei.value.status == gb.ERR_INVALID

"""fp64 CPU oracle for GraniKV decode-step attention.  TEST INFRASTRUCTURE ONLY.

Only the tests, the package's smoke check and the benchmark's CPU-baseline leg may import
this module.  The product path never calls it.

What it computes (GraniKV, "Ethics Statement": the layer changes memory layout and kernel
choice, not outputs; "2 Related Work", prefix-suffix attention: the prefix and suffix
partial attentions are merged with log-sum-exp).  So the exact result is ordinary softmax
attention of each decode query over its request's logical key sequence, which is the shared
prefix followed by the request's own suffix and decoded tokens:

    s_t  = scale * <q_{b,h}, K_b[t, j]>           j = h // (n_q / n_kv)  (grouped-query heads)
    lse  = m + ln sum_t exp(s_t - m),   m = max_t s_t
    o    = sum_t exp(s_t - lse) * V_b[t, j]

with ``scale = 1/sqrt(d)``.  Everything runs in float64 on a flat per-request copy built from
the workload's logical arrays, never from a KV pool, so a gather or slot error on the GPU
shows up as a value error.

An empty key sequence gives the empty partial (o = 0, lse = -inf); merging with it is the
identity.  Parity of every function here is pinned by tests/test_oracle_pins.py (brute force,
closed forms, merge invariants, permutation invariance, planted needles; for causal_prefill,
PyTorch's causal scaled-dot-product attention, the one-key closed form of the first token and
the direction of the mask).
"""

from __future__ import annotations

import math
from typing import Iterable, List, Optional, Tuple

import numpy as np


def softmax_scale(d: int) -> float:
    """The softmax scale 1/sqrt(d) (the pages leave it to the model; this is the standard)."""
    return 1.0 / math.sqrt(d)


def kv_head(h: int, n_q: int, n_kv: int) -> int:
    """KV head serving query head h under grouped-query attention: consecutive groups of
    n_q/n_kv query heads share one KV head (the pages write M_eff = B * n_q/kv and say no
    more; contiguous grouping is the standard layout)."""
    return h // (n_q // n_kv)


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> Tuple[np.ndarray, float]:
    """Softmax attention of one query vector over L keys; returns (o[d], lse) in float64.

    q: [d]; K, V: [L, d].  L == 0 returns the empty partial (zeros, -inf).
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    if K.shape[0] == 0:
        return np.zeros(V.shape[1] if V.ndim == 2 else q.shape[0], dtype=np.float64), -math.inf
    s = scale * (K @ q)
    m = float(np.max(s))
    w = np.exp(s - m)
    z = float(np.sum(w))
    lse = m + math.log(z)
    o = (w / z) @ V
    return o, lse


def lse_merge(parts: Iterable[Tuple[np.ndarray, float]]) -> Tuple[np.ndarray, float]:
    """Merge partial attention states (o_i, lse_i) over disjoint key sets.

    lse = M + ln sum_i exp(lse_i - M) with M = max_i lse_i, and
    o   = sum_i exp(lse_i - lse) * o_i.
    Empty partials (lse = -inf) contribute nothing.  All empty -> (0, -inf).
    """
    parts = list(parts)
    lses = [p[1] for p in parts]
    finite = [x for x in lses if x != -math.inf]
    if not finite:
        return np.zeros_like(np.asarray(parts[0][0], dtype=np.float64)), -math.inf
    M = max(finite)
    tot = math.fsum(math.exp(x - M) for x in finite)
    lse = M + math.log(tot)
    o = np.zeros_like(np.asarray(parts[0][0], dtype=np.float64))
    for oi, li in parts:
        if li != -math.inf:
            o = o + math.exp(li - lse) * np.asarray(oi, dtype=np.float64)
    return o, lse


def logical_kv(wl, b: int) -> Tuple[np.ndarray, np.ndarray]:
    """Request b's logical key/value sequence [L, n_kv, d] in float64: prefix then suffix.

    Built from the workload's logical arrays (the prefix as drawn, the suffix as drawn),
    independent of where the tokens are stored (HOT slab, COLD copy, slot order).
    """
    s = wl.spec
    parts_k, parts_v = [], []
    p = s.req_prefix[b]
    if p >= 0:
        parts_k.append(wl.prefix_k(p))
        parts_v.append(wl.prefix_v(p))
    parts_k.append(wl.suffix_k(b))
    parts_v.append(wl.suffix_v(b))
    K = np.concatenate(parts_k, axis=0).astype(np.float64)
    V = np.concatenate(parts_v, axis=0).astype(np.float64)
    return K, V


def request_attention(wl, b: int, heads: Optional[List[int]] = None):
    """Exact attention for request b: (o[len(heads), d], lse[len(heads)]) in float64."""
    s = wl.spec
    scale = softmax_scale(s.d)
    heads = list(range(s.n_q)) if heads is None else list(heads)
    K, V = logical_kv(wl, b)
    q = wl.q[b].astype(np.float64)
    o = np.zeros((len(heads), s.d), dtype=np.float64)
    lse = np.zeros(len(heads), dtype=np.float64)
    for i, h in enumerate(heads):
        j = kv_head(h, s.n_q, s.n_kv)
        o[i], lse[i] = attend(q[h], K[:, j, :], V[:, j, :], scale)
    return o, lse


def decode_attention(wl, requests: Optional[List[int]] = None):
    """Exact decode-step attention for the listed requests (default: all).

    Returns (o[R, n_q, d], lse[R, n_q]) in float64.
    """
    s = wl.spec
    requests = list(range(s.B)) if requests is None else list(requests)
    o = np.zeros((len(requests), s.n_q, s.d), dtype=np.float64)
    lse = np.zeros((len(requests), s.n_q), dtype=np.float64)
    for r, b in enumerate(requests):
        o[r], lse[r] = request_attention(wl, b)
    return o, lse


def prefix_suffix_partials(wl, b: int, h: int):
    """The two partial states of "2 Related Work" (prefix-suffix attention) for one row:
    ((o_p, lse_p), (o_s, lse_s)), either of which may be empty."""
    s = wl.spec
    j = kv_head(h, s.n_q, s.n_kv)
    scale = softmax_scale(s.d)
    q = wl.q[b, h].astype(np.float64)
    p = s.req_prefix[b]
    if p >= 0:
        pp = attend(q, wl.prefix_k(p)[:, j, :], wl.prefix_v(p)[:, j, :], scale)
    else:
        pp = (np.zeros(s.d), -math.inf)
    ss = attend(q, wl.suffix_k(b)[:, j, :], wl.suffix_v(b)[:, j, :], scale)
    return pp, ss


def causal_prefill(q: np.ndarray, K: np.ndarray, V: np.ndarray, tokens: Optional[List[int]] = None,
                   heads: Optional[List[int]] = None):
    """Causal self-attention of a prefix's own tokens, the step that fills a HOT slab
    ("2 Related Work", prefix-aware serving: a prefix is prefilled once, then reused): query
    token t attends keys 0..t of the prefix.

    q: [L, n_q, d]; K, V: [L, n_kv, d].  Returns (o [len(tokens), len(heads), d],
    lse [len(tokens), len(heads)]) in float64 for the requested tokens and heads (all by
    default), each one attend() over the first t+1 keys of its KV head."""
    L, n_q, d = q.shape
    n_kv = K.shape[1]
    tokens = list(range(L)) if tokens is None else list(tokens)
    heads = list(range(n_q)) if heads is None else list(heads)
    scale = softmax_scale(d)
    o = np.zeros((len(tokens), len(heads), d), dtype=np.float64)
    lse = np.zeros((len(tokens), len(heads)), dtype=np.float64)
    for a, t in enumerate(tokens):
        for c, h in enumerate(heads):
            j = kv_head(h, n_q, n_kv)
            o[a, c], lse[a, c] = attend(q[t, h], K[:t + 1, j], V[:t + 1, j], scale)
    return o, lse

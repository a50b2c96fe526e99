"""Pins for the CPU oracle: checks against things other than the oracle itself.

The GraniKV pages print no worked numeric example, so attention values are pinned by the
mathematics: arbitrary-precision brute force on tiny inputs, closed forms, the log-sum-exp
merge decomposition ("2 Related Work", prefix-suffix attention), invariance under token
permutation, and planted needles.  The pools are pinned by hand-derived scenarios in
tests/golden/ and the dispatch rule by hand-computed cells ("3 GraniKV", per-step dispatch).

The last test plants plausible mistakes in the oracle (on the CPU) and checks that at least
one pin catches each of them.
"""

import math
import os

import numpy as np
import pytest

import oracle.attention as A
import oracle.allocators as AL
import oracle.dispatch as D
from workloads import WorkloadSpec, Workload, small_mixed, tiny_fp32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


class _FakeWL:
    """Minimal stand-in for a Workload with hand-set arrays."""

    def __init__(self, n_q, n_kv, d, prefixes, req_prefix, suffixes, q):
        self.spec = WorkloadSpec(name="fake", dtype="f32", n_q=n_q, n_kv=n_kv, d=d,
                                 prefix_lens=[p[0].shape[0] for p in prefixes],
                                 req_prefix=list(req_prefix),
                                 suffix_lens=[s[0].shape[0] for s in suffixes],
                                 q_scale=1.0, n_slots=1 << 16)
        self._p = prefixes
        self._s = suffixes
        self.q = q

    def prefix_k(self, i):
        return self._p[i][0]

    def prefix_v(self, i):
        return self._p[i][1]

    def suffix_k(self, b):
        return self._s[b][0]

    def suffix_v(self, b):
        return self._s[b][1]


# ------------------------------------------------------------------------------------------
# attention pins (functions so that the mutation test can re-run them)

def pin_bruteforce_mpmath():
    """attend() == direct definition o = sum e^{s_t} v_t / sum e^{s_t}, lse = ln sum e^{s_t},
    evaluated without the max shift at 50 significant digits."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    rng = np.random.default_rng(1234)
    for trial in range(40):
        L = int(rng.integers(1, 9))
        d = int(rng.integers(1, 7))
        q = rng.standard_normal(d) * 2
        K = rng.standard_normal((L, d)) * 2
        V = rng.standard_normal((L, d))
        scale = 1.0 / math.sqrt(d)
        o, lse = A.attend(q, K, V, A.softmax_scale(d))
        s = [mp.mpf(scale) * mp.fsum(mp.mpf(float(q[i])) * mp.mpf(float(K[t, i])) for i in range(d))
             for t in range(L)]
        e = [mp.e ** st for st in s]
        z = mp.fsum(e)
        assert abs(float(mp.log(z)) - lse) <= 1e-12 * max(1.0, abs(lse))
        for i in range(d):
            ref = mp.fsum(e[t] * mp.mpf(float(V[t, i])) for t in range(L)) / z
            assert abs(float(ref) - o[i]) <= 1e-12


def pin_torch_softmax():
    """attend() == torch.softmax in float64 on small random inputs."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    for _ in range(20):
        L = int(rng.integers(1, 40))
        d = 16
        q = rng.standard_normal(d)
        K = rng.standard_normal((L, d))
        V = rng.standard_normal((L, d))
        sc = 1.0 / math.sqrt(d)
        o, lse = A.attend(q, K, V, A.softmax_scale(d))
        s = torch.from_numpy(K) @ torch.from_numpy(q) * sc
        p = torch.softmax(s, dim=0)
        o_ref = (p @ torch.from_numpy(V)).numpy()
        assert np.max(np.abs(o - o_ref)) <= 1e-12
        assert abs(lse - float(torch.logsumexp(s, dim=0))) <= 1e-12


def pin_closed_forms():
    rng = np.random.default_rng(3)
    d = 8
    sc = 1.0 / math.sqrt(d)
    q = rng.standard_normal(d)
    # L = 1: o = v, lse = s
    k = rng.standard_normal((1, d))
    v = rng.standard_normal((1, d))
    o, lse = A.attend(q, k, v, A.softmax_scale(d))
    assert np.allclose(o, v[0], atol=1e-14, rtol=0)
    assert abs(lse - sc * float(k[0] @ q)) <= 1e-13
    # all keys equal: o = mean(V), lse = s + ln L
    L = 7
    K = np.tile(k, (L, 1))
    V = rng.standard_normal((L, d))
    o, lse = A.attend(q, K, V, A.softmax_scale(d))
    assert np.allclose(o, V.mean(axis=0), atol=1e-13, rtol=0)
    assert abs(lse - (sc * float(k[0] @ q) + math.log(L))) <= 1e-12
    # constant V: o = V
    K = rng.standard_normal((L, d)) * 3
    V = np.tile(rng.standard_normal((1, d)), (L, 1))
    o, _ = A.attend(q, K, V, A.softmax_scale(d))
    assert np.allclose(o, V[0], atol=1e-13, rtol=0)
    # two keys: weights are the logistic function of the logit difference
    x = 1.7
    K2 = np.zeros((2, d))
    K2[1, 0] = x
    q2 = np.zeros(d)
    q2[0] = 1.0
    V2 = np.array([[1.0] + [0.0] * (d - 1), [0.0, 1.0] + [0.0] * (d - 2)])
    o, lse = A.attend(q2, K2, V2, A.softmax_scale(d))
    w1 = 1.0 / (1.0 + math.exp(-sc * x))
    assert abs(o[1] - w1) <= 1e-14 and abs(o[0] - (1 - w1)) <= 1e-14
    assert abs(lse - math.log(1.0 + math.exp(sc * x))) <= 1e-14
    # empty key set: the empty partial
    o, lse = A.attend(q, np.zeros((0, d)), np.zeros((0, d)), A.softmax_scale(d))
    assert lse == -math.inf and not np.any(o)


def pin_uniform_q_zero():
    rng = np.random.default_rng(5)
    d, L = 6, 11
    V = rng.standard_normal((L, d))
    o, lse = A.attend(np.zeros(d), rng.standard_normal((L, d)), V, A.softmax_scale(d))
    assert np.allclose(o, V.mean(axis=0), atol=1e-13, rtol=0)
    assert abs(lse - math.log(L)) <= 1e-13


def pin_gqa_mapping():
    """V constant = j+1 on KV head j  =>  o[b, h] = kv_head(h)+1 = h // (n_q/n_kv) + 1."""
    n_q, n_kv, d = 12, 3, 4
    rng = np.random.default_rng(11)
    Lp, Ls = 5, 4
    pk = rng.standard_normal((Lp, n_kv, d))
    pv = np.zeros((Lp, n_kv, d))
    sk = rng.standard_normal((Ls, n_kv, d))
    sv = np.zeros((Ls, n_kv, d))
    for j in range(n_kv):
        pv[:, j, :] = j + 1
        sv[:, j, :] = j + 1
    q = rng.standard_normal((1, n_q, d))
    wl = _FakeWL(n_q, n_kv, d, [(pk, pv)], [0], [(sk, sv)], q)
    o, _ = A.decode_attention(wl)
    for h in range(n_q):
        assert np.allclose(o[0, h], h // (n_q // n_kv) + 1, atol=1e-13, rtol=0)


def pin_concat_prefix_suffix():
    """q = 0: uniform weights over prefix+suffix, so o = (L_p a + L_s c)/(L_p+L_s) and
    lse = ln(L_p+L_s) when the prefix's V is a and the suffix's V is c; a request without a
    prefix averages its suffix only."""
    n_q, n_kv, d = 4, 2, 3
    rng = np.random.default_rng(13)
    Lp = 9
    pv = np.full((Lp, n_kv, d), 2.0)
    pk = rng.standard_normal((Lp, n_kv, d))
    suff = []
    lens = [4, 1, 6]
    for L in lens:
        suff.append((rng.standard_normal((L, n_kv, d)), np.full((L, n_kv, d), -1.0)))
    q = np.zeros((3, n_q, d))
    wl = _FakeWL(n_q, n_kv, d, [(pk, pv)], [0, 0, -1], suff, q)
    o, lse = A.decode_attention(wl)
    for b, L in enumerate(lens):
        lp = Lp if b < 2 else 0
        exp_o = (lp * 2.0 + L * -1.0) / (lp + L)
        assert np.allclose(o[b], exp_o, atol=1e-13, rtol=0)
        assert np.allclose(lse[b], math.log(lp + L), atol=1e-13, rtol=0)


def pin_merge_invariant():
    """Merging partials over any split of the keys equals attention over all keys; merging is
    associative and the empty partial is its identity."""
    rng = np.random.default_rng(17)
    d = 16
    for trial in range(20):
        L = int(rng.integers(2, 200))
        q = rng.standard_normal(d) * 1.5
        K = rng.standard_normal((L, d))
        V = rng.standard_normal((L, d))
        sc = A.softmax_scale(d)
        full = A.attend(q, K, V, sc)
        cuts = sorted(set(int(x) for x in rng.integers(0, L + 1, size=int(rng.integers(1, 6)))))
        bounds = [0] + cuts + [L]
        parts = [A.attend(q, K[a:b], V[a:b], sc) for a, b in zip(bounds[:-1], bounds[1:])]
        m = A.lse_merge(parts)
        assert np.max(np.abs(m[0] - full[0])) <= 1e-12 and abs(m[1] - full[1]) <= 1e-12
        if len(parts) >= 3:
            left = A.lse_merge([A.lse_merge(parts[:2])] + parts[2:])
            assert np.max(np.abs(left[0] - full[0])) <= 1e-12 and abs(left[1] - full[1]) <= 1e-12
        e = A.lse_merge([full, (np.zeros(d), -math.inf)])
        assert np.max(np.abs(e[0] - full[0])) <= 1e-15 and e[1] == full[1]


def pin_prefix_suffix_decomposition():
    """Merge of the prefix-only and suffix-only partials equals the full request attention."""
    wl = small_mixed(seed=2, dtype="f32", n_q=8, n_kv=2, d=32)
    for b in range(wl.spec.B):
        o, lse = A.request_attention(wl, b)
        for h in range(wl.spec.n_q):
            m = A.lse_merge(A.prefix_suffix_partials(wl, b, h))
            assert np.max(np.abs(m[0] - o[h])) <= 1e-12 and abs(m[1] - lse[h]) <= 1e-12


def pin_permutation_invariance():
    rng = np.random.default_rng(19)
    d, L = 16, 57
    q = rng.standard_normal(d)
    K = rng.standard_normal((L, d))
    V = rng.standard_normal((L, d))
    o, lse = A.attend(q, K, V, A.softmax_scale(d))
    perm = rng.permutation(L)
    o2, lse2 = A.attend(q, K[perm], V[perm], A.softmax_scale(d))
    assert np.max(np.abs(o - o2)) <= 1e-13 and abs(lse - lse2) <= 1e-13


def pin_needles():
    """A planted key with logit far above the rest takes > 99% of the weight: o ~= v_needle."""
    needles = [(0, 17, 3, 30.0), (1, 1005, 0, 30.0), (4, 250, 7, 30.0), (6, 100, 5, 30.0)]
    wl = small_mixed(seed=4, dtype="f32", needles=needles)
    for (b, pos, j, _) in needles:
        o, _ = A.request_attention(wl, b)
        K, V = A.logical_kv(wl, b)
        g = wl.spec.g
        for h in range(j * g, (j + 1) * g):
            assert np.max(np.abs(o[h] - V[pos, j])) <= 0.05, (b, h)


# ------------------------------------------------------------------------------------------
# causal prefill of a prefix (the step that fills a HOT slab)

def _prefill_case(L, n_q, n_kv, d, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((L, n_q, d))
    K = rng.standard_normal((L, n_kv, d))
    V = rng.standard_normal((L, n_kv, d))
    return q, K, V


def pin_prefill_torch_sdpa():
    # PyTorch's own causal scaled-dot-product attention in float64, KV heads repeated for GQA
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    for (L, n_q, n_kv, d) in [(37, 8, 2, 16), (64, 4, 4, 8), (9, 6, 1, 32)]:
        q, K, V = _prefill_case(L, n_q, n_kv, d, L)
        o, _ = A.causal_prefill(q, K, V)
        g = n_q // n_kv
        tq = torch.from_numpy(q).permute(1, 0, 2)                              # [n_q, L, d]
        tk = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(g, dim=0)  # [n_q, L, d]
        tv = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(g, dim=0)
        ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True).permute(1, 0, 2).numpy()
        assert np.max(np.abs(o - ref)) < 1e-12


def pin_prefill_first_token():
    # a single key: the output is that key's value row, the lse its scaled score
    q, K, V = _prefill_case(20, 8, 2, 16, 3)
    o, lse = A.causal_prefill(q, K, V, tokens=[0])
    for h in range(8):
        j = h // 4
        assert np.array_equal(o[0, h], V[0, j])
        assert abs(lse[0, h] - float(q[0, h] @ K[0, j]) / 4.0) < 1e-12


def pin_prefill_mask_direction():
    # token t does not see tokens after it, and does see the ones before it
    q, K, V = _prefill_case(30, 4, 2, 8, 5)
    o, lse = A.causal_prefill(q, K, V)
    K2, V2 = K.copy(), V.copy()
    K2[20:] += 3.0
    V2[20:] -= 2.0
    o2, lse2 = A.causal_prefill(q, K2, V2)
    assert np.array_equal(o[:20], o2[:20]) and np.array_equal(lse[:20], lse2[:20])
    assert np.all(np.abs(o[20:] - o2[20:]).max(axis=(1, 2)) > 1e-3)
    V3 = V.copy()
    V3[0] += 1.0
    o3, _ = A.causal_prefill(q, K, V3)
    assert np.all(np.abs(o3 - o).max(axis=(1, 2)) > 1e-6)


PINS = [pin_bruteforce_mpmath, pin_torch_softmax, pin_closed_forms, pin_uniform_q_zero,
        pin_gqa_mapping, pin_concat_prefix_suffix, pin_merge_invariant,
        pin_prefix_suffix_decomposition, pin_permutation_invariance, pin_needles,
        pin_prefill_torch_sdpa, pin_prefill_first_token, pin_prefill_mask_direction]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_attention_pin(pin):
    pin()


# ------------------------------------------------------------------------------------------
# pool pins

def _run_hot_scenario(path):
    hot = None
    with open(path) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "pool":
                hot = AL.HotFirstFit(int(tok[1]), max_slabs=int(tok[2]))
            elif tok[0] == "alloc":
                L = int(tok[1])
                want = tok[3:]
                if want == ["NO_HOT_SPACE"]:
                    with pytest.raises(AL.NoHotSpace):
                        hot.alloc(L)
                else:
                    assert hot.alloc(L) == (int(want[0]), int(want[1])), line
            elif tok[0] == "free":
                hot.free_slab(int(tok[1]))
            else:
                raise ValueError(line)


def _run_cold_scenario(path):
    ring = None
    tables = None
    with open(path) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "ring":
                ring = AL.ColdRing([int(x) for x in tok[1:]])
                tables = [[] for _ in range(3)]
            elif tok[0] == "alloc":
                arrow = tok.index("->")
                n_new = [int(x) for x in tok[1:arrow]]
                want = tok[arrow + 1:]
                if want == ["NO_COLD_SPACE"]:
                    before = (ring.head, ring.tail, [list(t) for t in tables])
                    with pytest.raises(AL.NoColdSpace):
                        ring.alloc(n_new, tables)
                    assert (ring.head, ring.tail, tables) == before
                else:
                    assert ring.alloc(n_new, tables) == [int(x) for x in want], line
            elif tok[0] == "free":
                ring.free([int(x) for x in tok[1:]])
            elif tok[0] == "table":
                b = int(tok[1])
                assert tables[b] == [int(x) for x in tok[3:]], line
            else:
                raise ValueError(line)


def test_hot_golden_scenario():
    _run_hot_scenario(os.path.join(GOLDEN, "hot_first_fit_scenario.txt"))


def test_cold_golden_scenario():
    _run_cold_scenario(os.path.join(GOLDEN, "cold_ring_scenario.txt"))


def test_hot_without_frees_is_a_bump_pointer():
    hot = AL.HotFirstFit(10_000)
    off = 0
    rng = np.random.default_rng(0)
    for i in range(20):
        L = int(rng.integers(1, 400))
        sid, o = hot.alloc(L)
        assert (sid, o) == (i, off)
        off += L


def test_hot_random_invariants():
    rng = np.random.default_rng(1)
    hot = AL.HotFirstFit(5000, max_slabs=64)
    for step in range(2000):
        if hot.slabs and rng.random() < 0.4:
            sid = int(rng.choice(list(hot.slabs)))
            hot.free_slab(sid)
        else:
            L = int(rng.integers(1, 800))
            try:
                sid, off = hot.alloc(L)
                assert 0 <= off and off + L <= 5000
            except AL.NoHotSpace:
                assert hot.largest_free() < L or len(hot.slabs) == 64
        # slabs and free extents tile [0, n_hot) exactly, extents are coalesced
        spans = sorted(list(hot.slabs.values()) + [tuple(e) for e in hot.free])
        pos = 0
        for o, ln in spans:
            assert o == pos and ln > 0
            pos += ln
        assert pos == 5000
        for a, b in zip(hot.free[:-1], hot.free[1:]):
            assert a[0] + a[1] < b[0]


def test_cold_ring_page_size_one_no_waste():
    """Page size 1: slots in use equal tokens stored, and no slot is handed out twice."""
    rng = np.random.default_rng(2)
    wl = tiny_fp32(seed=0)
    ring = AL.ColdRing(wl.cold_order)
    B = 4
    tables = [[] for _ in range(B)]
    for r in wl.append_schedule:
        ring.alloc(list(r), tables)
    used = [s for t in tables for s in t]
    assert len(used) == len(set(used)) == sum(wl.cold_len(b) for b in range(B))
    assert ring.n_free == ring.capacity - len(used)
    assert all(wl.spec.n_hot <= s < wl.spec.n_slots for s in used)


# ------------------------------------------------------------------------------------------
# dispatch pins

def test_dispatch_rule_hand_cells():
    # M_eff = B * n_q / n_kv, dense iff M_eff >= M_sat (inclusive), Llama shape g = 4
    assert D.m_eff(256, 32, 8) == 1024
    assert D.plan_groups([0] * 256, 32, 8, 1024)[0]["backend"] == D.DENSE
    assert D.plan_groups([0] * 255, 32, 8, 1024)[0]["backend"] == D.CASCADE
    # Qwen shape at TP=1, g = 5: B = 128 -> 640
    assert D.plan_groups([3] * 128, 40, 8, 640)[0]["backend"] == D.DENSE
    assert D.plan_groups([3] * 128, 40, 8, 641)[0]["backend"] == D.CASCADE
    # per-slab groups in order of first appearance; requests without a HOT prefix form none
    g = D.plan_groups([1, 0, 1, -1, 0, 0], 32, 8, 12)
    assert [x["slab"] for x in g] == [1, 0]
    assert [x["requests"] for x in g] == [[0, 2], [1, 4, 5]]
    assert [x["m_eff"] for x in g] == [8, 12]
    assert [x["backend"] for x in g] == [D.CASCADE, D.DENSE]


# ------------------------------------------------------------------------------------------
# planted mistakes: each must be caught by at least one pin

def _mut_scale_ignored(q, K, V, scale, _orig=A.attend):
    return _orig(q, K, V, 1.0)


def _mut_kv_swapped(q, K, V, scale, _orig=A.attend):
    return _orig(q, V, K, scale)


def _mut_drop_last(q, K, V, scale, _orig=A.attend):
    if len(K) > 1:
        return _orig(q, K[:-1], V[:-1], scale)
    return _orig(q, K, V, scale)


def _mut_lse_no_max(q, K, V, scale):
    q = np.asarray(q, float)
    K = np.asarray(K, float)
    V = np.asarray(V, float)
    if K.shape[0] == 0:
        return np.zeros(V.shape[1]), -math.inf
    s = scale * (K @ q)
    m = float(np.max(s))
    w = np.exp(s - m)
    return (w / w.sum()) @ V, math.log(w.sum())


def _mut_prefill_excludes_self(q, K, V, tokens=None, heads=None):
    L, n_q, d = q.shape
    tokens = list(range(L)) if tokens is None else list(tokens)
    heads = list(range(n_q)) if heads is None else list(heads)
    o = np.zeros((len(tokens), len(heads), d))
    lse = np.zeros((len(tokens), len(heads)))
    for a, t in enumerate(tokens):
        for c, h in enumerate(heads):
            j = A.kv_head(h, n_q, K.shape[1])
            o[a, c], lse[a, c] = A.attend(q[t, h], K[:t, j], V[:t, j], A.softmax_scale(d))
    return o, lse


def _mut_prefill_sees_next(q, K, V, tokens=None, heads=None):
    L, n_q, d = q.shape
    tokens = list(range(L)) if tokens is None else list(tokens)
    heads = list(range(n_q)) if heads is None else list(heads)
    o = np.zeros((len(tokens), len(heads), d))
    lse = np.zeros((len(tokens), len(heads)))
    for a, t in enumerate(tokens):
        for c, h in enumerate(heads):
            j = A.kv_head(h, n_q, K.shape[1])
            o[a, c], lse[a, c] = A.attend(q[t, h], K[:t + 2, j], V[:t + 2, j], A.softmax_scale(d))
    return o, lse


MUTATIONS = {
    "prefill_excludes_own_token": ("causal_prefill", _mut_prefill_excludes_self),
    "prefill_sees_next_token": ("causal_prefill", _mut_prefill_sees_next),
    "scale_ignored": ("attend", _mut_scale_ignored),
    "k_v_swapped": ("attend", _mut_kv_swapped),
    "last_token_dropped": ("attend", _mut_drop_last),
    "lse_missing_max": ("attend", _mut_lse_no_max),
    "gqa_modulo_mapping": ("kv_head", lambda h, n_q, n_kv: h % n_kv),
    "scale_1_over_d": ("softmax_scale", lambda d: 1.0 / d),
    "prefix_dropped": ("logical_kv", None),
    "merge_lse_is_max": ("lse_merge", None),
    "merge_unnormalised": ("lse_merge", None),
}


def _make_mutation(name):
    target, fn = MUTATIONS[name]
    if fn is not None:
        return target, fn
    if name == "prefix_dropped":
        def fn(wl, b, _orig=A.logical_kv):
            K, V = _orig(wl, b)
            L = wl.spec.suffix_lens[b]
            return K[K.shape[0] - L:], V[V.shape[0] - L:]
        return target, fn
    orig = A.lse_merge
    if name == "merge_lse_is_max":
        def fn(parts):
            parts = list(parts)
            o, lse = orig(parts)
            finite = [p[1] for p in parts if p[1] != -math.inf]
            return o, (max(finite) if finite else lse)
        return target, fn
    if name == "merge_unnormalised":
        def fn(parts):
            parts = list(parts)
            finite = [p[1] for p in parts if p[1] != -math.inf]
            if not finite:
                return orig(parts)
            M = max(finite)
            o = sum(math.exp(l - M) * np.asarray(x, float) for x, l in parts if l != -math.inf)
            return o, orig(parts)[1]
        return target, fn
    raise KeyError(name)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    target, fn = _make_mutation(name)
    monkeypatch.setattr(A, target, fn)
    caught = []
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            caught.append(pin.__name__)
        except pytest.skip.Exception:
            pass
    assert caught, f"no pin caught the planted mistake {name}"

"""Seeded synthetic workloads shaped like the GraniKV pages' decode workloads.

GraniKV (arXiv:2608.15584) evaluates decode over one long shared prefix (L_p up to 16K) plus
per-request suffixes drawn from ShareGPT-V3 traffic, and over several distinct prefixes of
mixed length ("B.8 Multi-prefix sensitivity").  The dataset is not available here, so these
generators stand in for it: every value is drawn from ``numpy.random.default_rng`` with a
fixed seed, and every length follows the stated distribution.

The module only draws numbers and arranges them.  It does no attention arithmetic: the
oracle and the CUDA path both consume a :class:`Workload` and neither depends on the other.

Random streams are keyed per object (``default_rng([seed, tag, index])``) so a single request
or prefix can be regenerated without drawing everything else; full-size cases can therefore be
checked on a sample of requests.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Callable, Dict, List, Optional, Sequence

import numpy as np

# Stream tags for default_rng([seed, tag, index]).
_TAG_STRUCT = 0
_TAG_PREFIX = 1
_TAG_SUFFIX = 2
_TAG_Q = 3
_TAG_COLD = 4
_TAG_SCHED = 5


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32.

    Inputs must be finite.  The result holds values exactly representable in bf16.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) >> 16) << 16
    return rounded.astype(np.uint32).view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Bit patterns (uint16) of float32 values that are already bf16-representable."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32)
    if np.any(bits & 0xFFFF):
        raise ValueError("bf16_bits: values are not bf16-representable; call round_to_bf16 first")
    return (bits >> 16).astype(np.uint16)


@dataclasses.dataclass
class WorkloadSpec:
    """Shape and structure of one decode step.

    ``req_prefix[b]`` is the index of request b's shared prefix (or -1 for none).
    ``prefix_in_hot[i]`` says whether prefix i was admitted to the HOT pool; a prefix that did
    not fit is stored per request at the head of each request's COLD token table (the paged
    fallback of "B.10 Cross-pool admission and promotion policy").
    """

    name: str
    dtype: str  # "f32" or "bf16"
    n_q: int
    n_kv: int
    d: int
    prefix_lens: List[int]
    req_prefix: List[int]
    suffix_lens: List[int]
    q_scale: float
    n_slots: int
    hot_fraction: float = 0.2
    prefix_in_hot: Optional[List[bool]] = None
    kv_scale: float = 1.0
    needles: List[tuple] = dataclasses.field(default_factory=list)  # (b, logical_pos, kv_head, score)
    schedule_max_chunk: int = 64

    def __post_init__(self):
        if self.dtype not in ("f32", "bf16"):
            raise ValueError("dtype must be f32 or bf16")
        if self.n_q % self.n_kv:
            raise ValueError("n_q must be a multiple of n_kv")
        if len(self.req_prefix) != len(self.suffix_lens):
            raise ValueError("req_prefix and suffix_lens differ in length")
        if self.prefix_in_hot is None:
            self.prefix_in_hot = [True] * len(self.prefix_lens)
        for b, (p, s) in enumerate(zip(self.req_prefix, self.suffix_lens)):
            if p < 0 and s == 0:
                raise ValueError(f"request {b} has neither prefix nor suffix")

    @property
    def B(self) -> int:
        return len(self.suffix_lens)

    @property
    def g(self) -> int:
        return self.n_q // self.n_kv

    @property
    def n_hot(self) -> int:
        return int(math.floor(self.hot_fraction * self.n_slots))


class Workload:
    """Materialises the random arrays of a :class:`WorkloadSpec` on demand.

    Logical arrays (what the oracle consumes):
      * ``q``                      [B, n_q, d]
      * ``prefix_k(i)/prefix_v(i)`` [L_p_i, n_kv, d]
      * ``suffix_k(b)/suffix_v(b)`` [L_s_b, n_kv, d]
    Storage layout helpers (what the GPU path consumes):
      * ``cold_len(b)``, ``cold_k(b)/cold_v(b)``: tokens request b keeps in COLD
        (a private prefix copy when its prefix is not in HOT, then its suffix)
      * ``cold_order``: initial COLD free-ring content, a seeded permutation of [n_hot, n_slots)
      * ``append_schedule``: rounds of per-request token counts appended to COLD, interleaved
        across requests so that consecutive tokens of one request land on unrelated slots.
    All float arrays are float32 holding values exact in the workload dtype.
    """

    def __init__(self, spec: WorkloadSpec, seed: int):
        self.spec = spec
        self.seed = int(seed)
        self._cache: Dict[tuple, np.ndarray] = {}

    # ---- random draws -------------------------------------------------------------------
    def _rng(self, tag: int, index: int = 0) -> np.random.Generator:
        return np.random.default_rng([self.seed, tag, index])

    def _normal(self, rng: np.random.Generator, shape, scale: float) -> np.ndarray:
        x = rng.standard_normal(shape, dtype=np.float32)
        if scale != 1.0:
            x = x * np.float32(scale)
        if self.spec.dtype == "bf16":
            x = round_to_bf16(x)
        return x

    def prefix_kv(self, i: int):
        key = ("p", i)
        if key not in self._cache:
            s = self.spec
            rng = self._rng(_TAG_PREFIX, i)
            k = self._normal(rng, (s.prefix_lens[i], s.n_kv, s.d), s.kv_scale)
            v = self._normal(rng, (s.prefix_lens[i], s.n_kv, s.d), s.kv_scale)
            self._cache[key] = (k, v)
            self._plant_needles()
        return self._cache[key]

    def suffix_kv(self, b: int):
        key = ("s", b)
        if key not in self._cache:
            s = self.spec
            rng = self._rng(_TAG_SUFFIX, b)
            k = self._normal(rng, (s.suffix_lens[b], s.n_kv, s.d), s.kv_scale)
            v = self._normal(rng, (s.suffix_lens[b], s.n_kv, s.d), s.kv_scale)
            self._cache[key] = (k, v)
            self._plant_needles()
        return self._cache[key]

    def prefix_k(self, i):
        return self.prefix_kv(i)[0]

    def prefix_v(self, i):
        return self.prefix_kv(i)[1]

    def suffix_k(self, b):
        return self.suffix_kv(b)[0]

    def suffix_v(self, b):
        return self.suffix_kv(b)[1]

    @property
    def q(self) -> np.ndarray:
        if "q" not in self._cache:
            s = self.spec
            self._cache["q"] = self._normal(self._rng(_TAG_Q), (s.B, s.n_q, s.d), s.q_scale)
        return self._cache["q"]

    def _plant_needles(self):
        """Overwrite planted keys: k = c * (sum of the group's query vectors), rounded.

        ``score`` is the target logit of the planted key for the group's heads (approximate;
        it ignores cross terms between the group's queries).  Input construction only.
        """
        s = self.spec
        for (b, pos, j, score) in s.needles:
            tag = ("needle", b, pos, j)
            if tag in self._cache:
                continue
            p = s.req_prefix[b]
            lp = s.prefix_lens[p] if p >= 0 else 0
            if pos < lp:
                key = ("p", p)
                row = pos
            else:
                key = ("s", b)
                row = pos - lp
            if key not in self._cache:
                continue  # planted when that array is drawn
            qsum = self.q[b, j * s.g:(j + 1) * s.g, :].astype(np.float64).sum(axis=0)
            qq = float(np.dot(self.q[b, j * s.g, :].astype(np.float64), qsum))
            c = score * math.sqrt(s.d) / max(qq, 1e-30)
            kvec = (c * qsum).astype(np.float32)
            if s.dtype == "bf16":
                kvec = round_to_bf16(kvec)
            self._cache[key][0][row, j, :] = kvec
            self._cache[tag] = np.zeros(0)

    # ---- layout helpers -----------------------------------------------------------------
    def logical_len(self, b: int) -> int:
        s = self.spec
        p = s.req_prefix[b]
        return (s.prefix_lens[p] if p >= 0 else 0) + s.suffix_lens[b]

    def hot_prefix(self, b: int) -> int:
        """Prefix index served from HOT for request b, or -1."""
        p = self.spec.req_prefix[b]
        return p if (p >= 0 and self.spec.prefix_in_hot[p]) else -1

    def cold_len(self, b: int) -> int:
        s = self.spec
        p = s.req_prefix[b]
        extra = s.prefix_lens[p] if (p >= 0 and not s.prefix_in_hot[p]) else 0
        return extra + s.suffix_lens[b]

    def cold_k(self, b: int) -> np.ndarray:
        return self._cold(b, 0)

    def cold_v(self, b: int) -> np.ndarray:
        return self._cold(b, 1)

    def _cold(self, b: int, which: int) -> np.ndarray:
        s = self.spec
        p = s.req_prefix[b]
        parts = []
        if p >= 0 and not s.prefix_in_hot[p]:
            parts.append(self.prefix_kv(p)[which])
        parts.append(self.suffix_kv(b)[which])
        return np.concatenate(parts, axis=0) if len(parts) > 1 else parts[0]

    @property
    def cold_order(self) -> np.ndarray:
        if "cold" not in self._cache:
            s = self.spec
            rng = self._rng(_TAG_COLD)
            self._cache["cold"] = (s.n_hot + rng.permutation(s.n_slots - s.n_hot)).astype(np.int32)
        return self._cache["cold"]

    @property
    def append_schedule(self) -> List[np.ndarray]:
        """Rounds of n_new[B]; round r appends n_new[b] tokens of request b, in request order."""
        if "sched" not in self._cache:
            s = self.spec
            rng = self._rng(_TAG_SCHED)
            remaining = np.array([self.cold_len(b) for b in range(s.B)], dtype=np.int64)
            rounds = []
            while remaining.sum() > 0:
                take = rng.integers(1, s.schedule_max_chunk + 1, size=s.B)
                skip = rng.random(s.B) < 0.25
                take[skip] = 0
                take = np.minimum(take, remaining)
                if take.sum() == 0:
                    continue
                rounds.append(take.astype(np.int32))
                remaining -= take
            self._cache["sched"] = rounds
        return self._cache["sched"]


def make_workload(spec: WorkloadSpec, seed: int) -> Workload:
    return Workload(spec, seed)


# ---- named recipes ----------------------------------------------------------------------------

def _lognormal_lens(rng, n, median=300.0, sigma=1.0, lo=32, hi=2048) -> List[int]:
    x = np.exp(rng.normal(math.log(median), sigma, size=n))
    return [int(v) for v in np.clip(np.rint(x), lo, hi)]


def _struct_rng(seed: int, name: str):
    return np.random.default_rng([int(seed), _TAG_STRUCT, sum(map(ord, name))])


def tiny_fp32(seed: int = 0) -> Workload:
    """fp32, n_q=8, n_kv=2, d=64, one HOT prefix of 256 tokens, B=4, suffixes U[16,64]."""
    rng = _struct_rng(seed, "tiny")
    B = 4
    spec = WorkloadSpec(
        name="tiny_fp32", dtype="f32", n_q=8, n_kv=2, d=64,
        prefix_lens=[256], req_prefix=[0] * B,
        suffix_lens=[int(x) for x in rng.integers(16, 65, size=B)],
        q_scale=1.0, n_slots=2048)
    return Workload(spec, seed)


def llama8b_single_prefix_16k(seed: int = 0, B: int = 64, q_scale: Optional[float] = None,
                              n_slots: int = 98304) -> Workload:
    """Llama-3.1-8B attention shape (32/8/128), bf16, one prefix of 16384 tokens, B=64,
    log-normal suffixes (median 300, sigma 1, clipped to [32, 2048]), q ~ N(0,1)/sqrt(128)."""
    rng = _struct_rng(seed, "llama")
    spec = WorkloadSpec(
        name="llama8b_single_prefix_16k", dtype="bf16", n_q=32, n_kv=8, d=128,
        prefix_lens=[16384], req_prefix=[0] * B, suffix_lens=_lognormal_lens(rng, B),
        q_scale=(1.0 / math.sqrt(128.0)) if q_scale is None else q_scale, n_slots=n_slots,
        schedule_max_chunk=512)
    return Workload(spec, seed)


def hetero_multi_prefix_k8(seed: int = 0, q_scale: Optional[float] = None) -> Workload:
    """k=8 distinct prefixes, L_p ~ U[2048,16384], 8-32 requests per prefix (total 160),
    log-normal suffixes; one mixed batch (requests of different prefixes interleaved)."""
    rng = _struct_rng(seed, "hetero")
    k = 8
    lps = [int(x) for x in rng.integers(2048, 16385, size=k)]
    counts = [8] * k
    for _ in range(160 - 8 * k):
        open_ = [i for i in range(k) if counts[i] < 32]
        counts[open_[int(rng.integers(0, len(open_)))]] += 1
    req_prefix = [i for i in range(k) for _ in range(counts[i])]
    req_prefix = [int(x) for x in rng.permutation(np.array(req_prefix))]
    B = len(req_prefix)
    hot_needed = sum(lps)
    n_slots = int(math.ceil(hot_needed / 0.2)) + 1024
    spec = WorkloadSpec(
        name="hetero_multi_prefix_k8", dtype="bf16", n_q=32, n_kv=8, d=128,
        prefix_lens=lps, req_prefix=req_prefix, suffix_lens=_lognormal_lens(rng, B),
        q_scale=(1.0 / math.sqrt(128.0)) if q_scale is None else q_scale, n_slots=n_slots,
        schedule_max_chunk=512)
    return Workload(spec, seed)


def qwen_tp1_16k(seed: int = 0, q_scale: Optional[float] = None) -> Workload:
    """Qwen-2.5-14B/32B attention shape at TP=1 (40/8/128), bf16, one prefix of 16384 tokens,
    B=128, suffixes U[64,1024].  KV budget 131072 slots: the COLD part (104,858 slots) holds the
    suffixes (about 70K tokens) and a few hundred decode steps of all 128 requests."""
    rng = _struct_rng(seed, "qwen")
    B = 128
    spec = WorkloadSpec(
        name="qwen_tp1_16k", dtype="bf16", n_q=40, n_kv=8, d=128,
        prefix_lens=[16384], req_prefix=[0] * B,
        suffix_lens=[int(x) for x in rng.integers(64, 1025, size=B)],
        q_scale=(1.0 / math.sqrt(128.0)) if q_scale is None else q_scale, n_slots=131072,
        schedule_max_chunk=512)
    return Workload(spec, seed)


def dispatch_sweep_cell(L_p: int, B: int, seed: int = 0, suffix_len: int = 256,
                        needles: Sequence[tuple] = ()) -> Workload:
    """One cell of the dense/cascade crossover sweep: Llama shape, one prefix, fixed suffix."""
    n_cold = B * suffix_len + 1024
    n_slots = max(int(math.ceil(L_p / 0.2)) + 8, int(math.ceil(n_cold / 0.8)) + 8)
    spec = WorkloadSpec(
        name=f"sweep_Lp{L_p}_B{B}", dtype="bf16", n_q=32, n_kv=8, d=128,
        prefix_lens=[L_p], req_prefix=[0] * B, suffix_lens=[suffix_len] * B,
        q_scale=1.0 / math.sqrt(128.0), n_slots=n_slots, schedule_max_chunk=suffix_len,
        needles=list(needles))
    return Workload(spec, seed)


def small_mixed(seed: int = 0, dtype: str = "bf16", n_q: int = 32, n_kv: int = 8, d: int = 128,
                q_scale: float = 1.0, needles: Sequence[tuple] = ()) -> Workload:
    """Small multi-tile case with ragged tails and the degenerate requests:

    * two HOT prefixes of ragged length and one prefix that did not fit in HOT (paged
      fallback: its tokens head each of its requests' COLD tables);
    * a request with a prefix and an empty suffix, and a request with no prefix at all;
    * suffix lengths that are not multiples of any tile size.
    """
    rng = _struct_rng(seed, "small" + dtype)
    lps = [1000, 333, 200]
    req_prefix = [0, 0, 1, 0, -1, 1, 2, 0, 2, 1]
    B = len(req_prefix)
    sl = [int(x) for x in rng.integers(1, 300, size=B)]
    sl[3] = 0      # prefix only
    sl[4] = 517    # no prefix, suffix only
    spec = WorkloadSpec(
        name=f"small_mixed_{dtype}", dtype=dtype, n_q=n_q, n_kv=n_kv, d=d,
        prefix_lens=lps, req_prefix=req_prefix, suffix_lens=sl, q_scale=q_scale,
        n_slots=8192, prefix_in_hot=[True, True, False], needles=list(needles),
        schedule_max_chunk=48)
    return Workload(spec, seed)


def medium_shared(seed: int = 0, B: int = 70, L_p: int = 3000, q_scale: float = 1.0,
                  needles: Sequence[tuple] = ()) -> Workload:
    """One ragged prefix shared by enough requests for several 128-row blocks (B*g rows, the
    last block partial) and several L_p pieces, plus short ragged suffixes."""
    rng = _struct_rng(seed, "medium")
    spec = WorkloadSpec(
        name="medium_shared", dtype="bf16", n_q=32, n_kv=8, d=128,
        prefix_lens=[L_p], req_prefix=[0] * B,
        suffix_lens=[int(x) for x in rng.integers(1, 100, size=B)],
        q_scale=q_scale, n_slots=32768, needles=list(needles), schedule_max_chunk=64)
    return Workload(spec, seed)


NAMED: Dict[str, Callable[..., Workload]] = {
    "tiny_fp32": tiny_fp32,
    "llama8b_single_prefix_16k": llama8b_single_prefix_16k,
    "hetero_multi_prefix_k8": hetero_multi_prefix_k8,
    "qwen_tp1_16k": qwen_tp1_16k,
    "small_mixed": small_mixed,
    "medium_shared": medium_shared,
}

"""Place a synthetic :class:`workloads.Workload` into a :class:`GraniKVCache` through the library's
own calls: HOT-first admission of each prefix, then the COLD appends of its schedule.

Layout only: values are copied as drawn (the generator already rounded them to the workload
dtype), so no arithmetic of the method happens here.
"""

from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np
import torch

from . import _binding as gb
from .cache import GraniKVCache


@dataclasses.dataclass
class LoadedWorkload:
    cache: GraniKVCache
    slab_ids: List[int]
    q: torch.Tensor
    batch: gb.Batch


def _dev(x: np.ndarray, dtype, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).to(device=device).to(dtype)


def load_workload(wl, *, n_layers: int = 1, device: int = 0, m_sat: int = 0, cap: Optional[int] = None,
                  cache: Optional[GraniKVCache] = None, layer_fill=None) -> LoadedWorkload:
    """Build a cache for ``wl`` (or reuse ``cache``) and load prefixes, COLD tokens and q.

    Every layer receives the workload's K/V unless ``layer_fill(layer, name, shape)`` supplies
    a tensor for layers > 0 (used by the benchmark to give each layer distinct data).
    """
    s = wl.spec
    dtype = gb.DTYPE_BF16 if s.dtype == "bf16" else gb.DTYPE_F32
    B = s.B
    cold_lens = [wl.cold_len(b) for b in range(B)]
    if cap is None:
        cap = max(64, ((max(cold_lens) + 64 + 63) // 64) * 64)
    if cache is None:
        cache = GraniKVCache(n_layers=n_layers, n_q=s.n_q, n_kv=s.n_kv, head_dim=s.d, dtype=dtype,
                             n_slots=s.n_slots, max_batch=B, cap=cap, hot_fraction=s.hot_fraction,
                             cold_init_order=wl.cold_order, m_sat=m_sat, device=device)
    tdt = cache.tdtype
    dev = cache.device

    def layers_of(arr_fn, shape):
        base = None
        out = []
        for layer in range(cache.n_layers):
            if layer > 0 and layer_fill is not None:
                out.append(layer_fill(layer, shape))
            else:
                if base is None:
                    base = _dev(arr_fn(), tdt, dev)
                out.append(base)
        return out

    used = sorted({p for p in s.req_prefix if p >= 0})
    slab_of = {}
    for i in used:
        if not s.prefix_in_hot[i]:
            continue
        shape = (s.prefix_lens[i], s.n_kv, s.d)
        ks = layers_of(lambda: wl.prefix_k(i), shape)
        vs = layers_of(lambda: wl.prefix_v(i), shape)
        sid = cache.admit_prefix(s.prefix_lens[i], ks, vs)
        if sid is None:
            raise gb.NoHotSpace(gb.ERR_NO_HOT_SPACE, "load_workload", f"prefix {i} does not fit in HOT")
        slab_of[i] = sid
    done = [0] * B
    for n_new in wl.append_schedule:
        parts_k, parts_v = [], []
        for b in range(B):
            n = int(n_new[b])
            if n:
                parts_k.append(wl.cold_k(b)[done[b]:done[b] + n])
                parts_v.append(wl.cold_v(b)[done[b]:done[b] + n])
                done[b] += n
        kk = np.concatenate(parts_k, axis=0)
        vv = np.concatenate(parts_v, axis=0)
        ks = layers_of(lambda: kk, kk.shape)
        vs = layers_of(lambda: vv, vv.shape)
        cache.append([int(x) for x in n_new], ks, vs)
    assert done == cold_lens
    q = _dev(wl.q, tdt, dev)
    slab_ids = [slab_of[p] if (p >= 0 and s.prefix_in_hot[p]) else -1 for p in s.req_prefix]
    batch = cache.batch(slab_ids)
    return LoadedWorkload(cache=cache, slab_ids=slab_ids, q=q, batch=batch)

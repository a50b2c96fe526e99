"""A GraniKV KV cache on one GPU: torch supplies the device memory and streams, libgranikv does
every step of the path (pools, slot allocation, K/V scatter, dispatch, attention, merge).

GraniKV (arXiv:2608.15584), "3 GraniKV": one KV buffer per layer split into a contiguous HOT
pool (one slab per shared prefix) and a token-level COLD pool (page size 1) for suffix and
decoded tokens; "B.10 Cross-pool admission and promotion policy": HOT first, COLD fallback.
"""

from __future__ import annotations

from typing import List, Optional, Sequence

import torch

from . import _binding as gb

_TORCH_DTYPE = {gb.DTYPE_F32: torch.float32, gb.DTYPE_BF16: torch.bfloat16}


class GraniKVCache:
    """Per-layer K/V pools [n_slots, n_kv, d], per-request COLD token tables, and a context."""

    def __init__(self, *, n_layers: int, n_q: int, n_kv: int, head_dim: int, dtype: int,
                 n_slots: int, max_batch: int, cap: int, hot_fraction: float = 0.2,
                 cold_init_order: Optional[Sequence[int]] = None, m_sat: int = 0,
                 device: int = 0, max_slabs: int = 0):
        if not torch.cuda.is_available():
            raise RuntimeError("GraniKVCache needs a CUDA device")
        self.device = torch.device("cuda", device)
        self.tdtype = _TORCH_DTYPE[dtype]
        self.n_layers, self.n_q, self.n_kv, self.head_dim = n_layers, n_q, n_kv, head_dim
        self.dtype, self.n_slots, self.cap, self.max_batch = dtype, n_slots, cap, max_batch
        self.k_pools: List[torch.Tensor] = []
        self.v_pools: List[torch.Tensor] = []
        for _ in range(n_layers):
            self.k_pools.append(torch.zeros((n_slots, n_kv, head_dim), dtype=self.tdtype, device=self.device))
            self.v_pools.append(torch.zeros((n_slots, n_kv, head_dim), dtype=self.tdtype, device=self.device))
        self.ctx = gb.Context(n_layers=n_layers, n_q=n_q, n_kv=n_kv, head_dim=head_dim, dtype=dtype,
                              n_slots=n_slots, k_pools=self.k_pools, v_pools=self.v_pools,
                              hot_fraction=hot_fraction, cold_init_order=cold_init_order,
                              m_sat=m_sat, max_batch=max_batch, device=device, max_slabs=max_slabs)
        self.req_to_slot = torch.zeros((max_batch, cap), dtype=torch.int32, device=self.device)
        self.suffix_len = torch.zeros((max_batch,), dtype=torch.int32, device=self.device)
        self.seq_len_host = [0] * max_batch
        self._ws: Optional[torch.Tensor] = None

    @property
    def n_hot(self) -> int:
        return self.ctx.hot_stats()[0]

    def stream(self):
        return torch.cuda.current_stream(self.device)

    # prefixes -----------------------------------------------------------------------------
    def admit_prefix(self, L_p: int, k_layers: Sequence[torch.Tensor], v_layers: Sequence[torch.Tensor]):
        """HOT-first admission: a slab id, or None when no HOT extent can hold L_p slots (the
        caller then stores the prefix in each request's COLD table)."""
        try:
            sid, _ = self.ctx.hot_alloc(L_p)
        except gb.NoHotSpace:
            return None
        s = self.stream()
        for layer in range(self.n_layers):
            k = k_layers[layer].contiguous()
            v = v_layers[layer].contiguous()
            self.ctx.hot_fill(layer, sid, k, v, s)
        return sid

    # COLD tokens --------------------------------------------------------------------------
    def append(self, n_new: Sequence[int], k_layers: Sequence[torch.Tensor], v_layers: Sequence[torch.Tensor],
               slots_out: Optional[torch.Tensor] = None) -> torch.Tensor:
        """Append n_new[b] tokens to request b (b < len(n_new)): pop COLD slots, then scatter each
        layer's new K/V ([sum n_new, n_kv, d], request order) into them.  Returns the slots."""
        B = len(n_new)
        N = int(sum(n_new))
        if slots_out is None:
            slots_out = torch.empty((max(N, 1),), dtype=torch.int32, device=self.device)
        s = self.stream()
        self.ctx.cold_alloc(list(n_new), self.req_to_slot, self.suffix_len, self.cap, slots_out, s)
        for b in range(B):
            self.seq_len_host[b] += int(n_new[b])
        if N:
            for layer in range(self.n_layers):
                self.ctx.cold_append(layer, k_layers[layer].contiguous(), v_layers[layer].contiguous(),
                                     slots_out, N, s)
        return slots_out[:N]

    # attention ----------------------------------------------------------------------------
    def batch(self, slab_ids: Sequence[int], seq_len: Optional[Sequence[int]] = None) -> gb.Batch:
        B = len(slab_ids)
        lens = list(seq_len) if seq_len is not None else self.seq_len_host[:B]
        return gb.Batch(slab_ids, lens, self.req_to_slot, self.cap)

    def workspace(self, plan: gb.Plan) -> torch.Tensor:
        n = self.ctx.workspace_size(plan)
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty((max(n, 256),), dtype=torch.uint8, device=self.device)
        return self._ws

    def decode(self, layer: int, q: torch.Tensor, batch: gb.Batch, plan: Optional[gb.Plan] = None,
               o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None):
        """Decode-step attention of q [B, n_q, d] for one layer; returns (o, lse)."""
        if plan is None:
            plan = self.ctx.dispatch(batch)
        B = batch.B
        if o is None:
            o = torch.empty((B, self.n_q, self.head_dim), dtype=self.tdtype, device=self.device)
        if lse is None:
            lse = torch.empty((B, self.n_q), dtype=torch.float32, device=self.device)
        ws = self.workspace(plan)
        self.ctx.decode_attention(layer, q, batch, plan, o, lse, ws, ws.numel(), self.stream())
        return o, lse

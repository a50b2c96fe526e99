"""A GraniKV KV cache on one GPU: torch supplies the device memory and streams, libgranikv does
every step of the path (pools, slot allocation, K/V scatter, dispatch, attention, merge).

GraniKV (arXiv:2608.15584), "3 GraniKV": one KV buffer per layer split into a contiguous HOT
pool (one slab per shared prefix) and a token-level COLD pool (page size 1) for suffix and
decoded tokens; "B.10 Cross-pool admission and promotion policy": HOT first, COLD fallback.
"""

from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple

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
        self._index: Optional[gb.Index] = None
        self.cached: Dict[int, dict] = {}                      # prefixes written by admit()
        self.cold_prefix_slots: Dict[int, torch.Tensor] = {}  # COLD-placed prefix -> its slots
        self.row_prefix: List[Optional[Tuple[int, int]]] = [None] * max_batch  # (handle, shared COLD len)

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

    # prefix lifecycle ("2 Related Work": a reference-counted radix index over token ids;
    # "B.10": HOT first, COLD fallback, no demotion) ---------------------------------------
    @property
    def index(self) -> gb.Index:
        if self._index is None:
            self._index = self.ctx.index()
        return self._index

    def admit(self, tokens: Sequence[int], k_layers: Sequence[torch.Tensor], v_layers: Sequence[torch.Tensor]):
        """Cache a prefix given by its token ids and its K/V per layer ([L_p, n_kv, d] each).
        HOT first (a slab filled by device copies); if the index places it in COLD, its K/V go
        once into COLD slots that the prefix owns and that its requests share.  Returns
        (prefix info, evicted handles); an already-cached prefix is not written again."""
        info, evicted = self.index.insert(tokens)
        for pid in evicted:  # only unreferenced HOT prefixes are evicted; their slabs are free
            self.cached.pop(pid, None)
        pid, L_p = info["prefix_id"], info["length"]
        if pid in self.cached:
            return info, evicted
        s = self.stream()
        if info["slab_id"] >= 0:
            for layer in range(self.n_layers):
                self.ctx.hot_fill(layer, info["slab_id"], k_layers[layer].contiguous(),
                                  v_layers[layer].contiguous(), s)
        else:
            table = torch.empty((1, L_p), dtype=torch.int32, device=self.device)
            count = torch.zeros((1,), dtype=torch.int32, device=self.device)
            slots = torch.empty((L_p,), dtype=torch.int32, device=self.device)
            self.ctx.cold_alloc([L_p], table, count, L_p, slots, s)
            for layer in range(self.n_layers):
                self.ctx.cold_append(layer, k_layers[layer].contiguous(), v_layers[layer].contiguous(),
                                     slots, L_p, s)
            self.cold_prefix_slots[pid] = slots
        self.cached[pid] = info
        return info, evicted

    def attach(self, b: int, tokens: Sequence[int]):
        """Start request row b from its prompt's token ids: the longest cached prefix it starts
        with is matched and referenced.  A HOT prefix is read through its slab; a COLD one's
        slots head the row's token table.  Returns (slab id or -1, prefix tokens reused); the
        caller then appends the remaining prompt tokens with append()."""
        if self.row_prefix[b] is not None or self.seq_len_host[b]:
            raise RuntimeError(f"row {b} is in use")
        info = self.index.match(tokens, acquire=True)
        pid = info["prefix_id"]
        if pid < 0:
            self.row_prefix[b] = None
            return -1, 0
        if info["slab_id"] >= 0:
            self.row_prefix[b] = (pid, 0)
            return info["slab_id"], info["length"]
        L_p = info["length"]
        if L_p > self.cap:
            self.index.release(pid)
            raise ValueError("a COLD prefix longer than the token table")
        self.req_to_slot[b, :L_p].copy_(self.cold_prefix_slots[pid])
        self.suffix_len[b].fill_(L_p)
        self.seq_len_host[b] = L_p
        self.row_prefix[b] = (pid, L_p)
        return -1, L_p

    def detach(self, b: int):
        """Request row b is finished: its own COLD slots return to the free ring and its prefix
        reference is dropped (the prefix stays cached until evicted or removed)."""
        shared = 0
        if self.row_prefix[b] is not None:
            pid, shared = self.row_prefix[b]
            self.index.release(pid)
        own = self.seq_len_host[b] - shared
        if own > 0:
            self.ctx.cold_free(self.req_to_slot[b, shared:self.seq_len_host[b]].clone(), own, self.stream())
        self.row_prefix[b] = None
        self.seq_len_host[b] = 0
        self.suffix_len[b].zero_()

    def remove_prefix(self, pid: int):
        """Drop an unreferenced cached prefix: a HOT slab returns to the pool, a COLD prefix's
        slots to the free ring."""
        self.index.remove(pid)
        self.cached.pop(pid, None)
        slots = self.cold_prefix_slots.pop(pid, None)
        if slots is not None:
            self.ctx.cold_free(slots, slots.numel(), self.stream())

    def move_row(self, src: int, dst: int):
        """Move request row src (token table, lengths, prefix reference) into the free row dst."""
        if src == dst:
            return
        self.req_to_slot[dst].copy_(self.req_to_slot[src])
        self.suffix_len[dst].copy_(self.suffix_len[src])
        self.seq_len_host[dst] = self.seq_len_host[src]
        self.row_prefix[dst] = self.row_prefix[src]
        self.seq_len_host[src] = 0
        self.row_prefix[src] = None
        self.suffix_len[src].zero_()

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

    def alloc(self, n_new: Sequence[int], slots_out: Optional[torch.Tensor] = None) -> torch.Tensor:
        """Pop n_new[b] COLD slots for request b (b < len(n_new)) into its token table, without
        writing K/V (decode() with k_new/v_new writes the step's new token).  Returns the slots."""
        N = int(sum(n_new))
        if slots_out is None:
            slots_out = torch.empty((max(N, 1),), dtype=torch.int32, device=self.device)
        self.ctx.cold_alloc(list(n_new), self.req_to_slot, self.suffix_len, self.cap, slots_out, self.stream())
        for b in range(len(n_new)):
            self.seq_len_host[b] += int(n_new[b])
        return slots_out[:N]

    @property
    def fused_append(self) -> bool:
        """decode() can write the step's new K/V itself (granikv_decode_attention_append), on
        every path of the library."""
        return True

    def decode(self, layer: int, q: torch.Tensor, batch: gb.Batch, plan: Optional[gb.Plan] = None,
               o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
               k_new: Optional[torch.Tensor] = None, v_new: Optional[torch.Tensor] = None):
        """Decode-step attention of q [B, n_q, d] for one layer; returns (o, lse).  With k_new and
        v_new ([B, n_kv, d]), row b is the K/V of request b's newest token (the last of its COLD
        list, slot already allocated): it is written to that slot by the same launches."""
        if plan is None:
            plan = self.ctx.dispatch(batch)
        B = batch.B
        if o is None:
            o = torch.empty((B, self.n_q, self.head_dim), dtype=self.tdtype, device=self.device)
        if lse is None:
            lse = torch.empty((B, self.n_q), dtype=torch.float32, device=self.device)
        ws = self.workspace(plan)
        if k_new is not None:
            self.ctx.decode_attention_append(layer, q, k_new.contiguous(), v_new.contiguous(), batch, plan, o, lse,
                                             ws, ws.numel(), self.stream())
        else:
            self.ctx.decode_attention(layer, q, batch, plan, o, lse, ws, ws.numel(), self.stream())
        return o, lse

    def prefill(self, layer: int, slab_id: int, q: torch.Tensor, k: Optional[torch.Tensor] = None,
                v: Optional[torch.Tensor] = None, o: Optional[torch.Tensor] = None,
                lse: Optional[torch.Tensor] = None):
        """Causal prefill of a HOT prefix in one layer: its K/V ([L_p, n_kv, d], if given) are
        written into the slab, then each of its L_p query tokens (q [L_p, n_q, d]) attends the
        slab up to itself.  Returns (o [L_p, n_q, d], lse [L_p, n_q])."""
        L_p = q.shape[0]
        if o is None:
            o = torch.empty((L_p, self.n_q, self.head_dim), dtype=self.tdtype, device=self.device)
        if lse is None:
            lse = torch.empty((L_p, self.n_q), dtype=torch.float32, device=self.device)
        n = self.ctx.prefill_workspace_size(L_p)
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty((max(n, 256),), dtype=torch.uint8, device=self.device)
        kk = k.contiguous() if k is not None else None
        vv = v.contiguous() if v is not None else None
        self.ctx.prefill_attention(layer, slab_id, kk, vv, q.contiguous(), o, lse, self._ws, self._ws.numel(),
                                   self.stream())
        return o, lse

"""ctypes binding of libgranikv (include/granikv.h): same entry points, argument marshalling only.

Device buffers are passed as integer addresses (or any object with ``data_ptr()``, such as a
torch tensor) and streams as integer ``cudaStream_t`` handles (or objects with a
``cuda_stream`` attribute).  Every step of the decode path runs in the library's CUDA
kernels; there is no fallback.  If the library has not been built, every call raises.
"""

from __future__ import annotations

import ctypes as C
import os
import weakref
from typing import Optional, Sequence

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgranikv.so")

OK = 0
ERR_INVALID = 1
ERR_NO_HOT_SPACE = 2
ERR_NO_COLD_SPACE = 3
ERR_CUDA = 4
ERR_DEVICE_CHECK = 5
ERR_UNSUPPORTED = 6
ERR_NO_DEVICE = 7
ERR_STATIC_WORKSPACE_TOO_SMALL = 8

DTYPE_F32 = 0
DTYPE_BF16 = 1

BACKEND_AUTO = 0
BACKEND_DENSE = 1
BACKEND_CASCADE = 2
BACKEND_NAMES = {BACKEND_AUTO: "auto", BACKEND_DENSE: "dense", BACKEND_CASCADE: "cascade"}


class GranikvError(RuntimeError):
    def __init__(self, status: int, where: str, text: str):
        super().__init__(f"{where}: {text} (status {status})")
        self.status = status


class NoHotSpace(GranikvError):
    pass


class NoColdSpace(GranikvError):
    pass


class DeviceCheckFailed(GranikvError):
    pass


class _Config(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("n_q", C.c_int32), ("n_kv", C.c_int32),
                ("head_dim", C.c_int32), ("dtype", C.c_int32), ("device", C.c_int32),
                ("n_slots", C.c_int64), ("hot_fraction", C.c_double),
                ("k_pool", C.POINTER(C.c_void_p)), ("v_pool", C.POINTER(C.c_void_p)),
                ("cold_init_order", C.POINTER(C.c_int32)), ("m_sat", C.c_int32),
                ("max_slabs", C.c_int32), ("max_batch", C.c_int32), ("host_only", C.c_int32)]


class _Batch(C.Structure):
    _fields_ = [("B", C.c_int32), ("slab_id", C.POINTER(C.c_int32)),
                ("seq_len", C.POINTER(C.c_int32)), ("req_to_slot", C.c_void_p), ("cap", C.c_int32),
                ("seq_len_dev", C.c_void_p)]


class GroupInfo(C.Structure):
    _fields_ = [("slab_id", C.c_int32), ("n_requests", C.c_int32), ("m_eff", C.c_int32),
                ("backend", C.c_int32), ("L_p", C.c_int32), ("n_splits", C.c_int32),
                ("slot_offset", C.c_int64)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class PrefixInfo(C.Structure):
    _fields_ = [("prefix_id", C.c_int32), ("length", C.c_int32), ("slab_id", C.c_int32),
                ("refcount", C.c_int32), ("slot_offset", C.c_int64)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


_lib = None

# (name, restype, argtypes) of every exported symbol
_SIGNATURES = [
    ("granikv_status_string", C.c_char_p, [C.c_int32]),
    ("granikv_version", C.c_int32, []),
    ("granikv_create", C.c_int32, [C.POINTER(_Config), C.POINTER(C.c_void_p)]),
    ("granikv_destroy", C.c_int32, [C.c_void_p]),
    ("granikv_hot_alloc", C.c_int32, [C.c_void_p, C.c_int32, C.POINTER(C.c_int32), C.POINTER(C.c_int64)]),
    ("granikv_hot_free", C.c_int32, [C.c_void_p, C.c_int32]),
    ("granikv_hot_info", C.c_int32, [C.c_void_p, C.c_int32, C.POINTER(C.c_int64), C.POINTER(C.c_int32)]),
    ("granikv_hot_stats", C.c_int32, [C.c_void_p, C.POINTER(C.c_int64), C.POINTER(C.c_int64)]),
    ("granikv_hot_fill", C.c_int32, [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p]),
    ("granikv_cold_alloc", C.c_int32, [C.c_void_p, C.POINTER(C.c_int32), C.c_int32, C.c_void_p,
                                       C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p]),
    ("granikv_cold_free", C.c_int32, [C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p]),
    ("granikv_cold_free_count", C.c_int32, [C.c_void_p, C.POINTER(C.c_int64)]),
    ("granikv_cold_alloc_uniform", C.c_int32, [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                                               C.c_int32, C.c_void_p, C.c_void_p]),
    ("granikv_cold_sync", C.c_int32, [C.c_void_p, C.c_void_p]),
    ("granikv_cold_append", C.c_int32, [C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p,
                                        C.c_int32, C.c_void_p]),
    ("granikv_index_create", C.c_int32, [C.c_void_p, C.POINTER(C.c_void_p)]),
    ("granikv_index_destroy", C.c_int32, [C.c_void_p]),
    ("granikv_index_match", C.c_int32, [C.c_void_p, C.POINTER(C.c_int32), C.c_int32, C.c_int32,
                                        C.POINTER(PrefixInfo)]),
    ("granikv_index_insert", C.c_int32, [C.c_void_p, C.POINTER(C.c_int32), C.c_int32, C.POINTER(PrefixInfo),
                                         C.POINTER(C.c_int32), C.c_int32, C.POINTER(C.c_int32)]),
    ("granikv_index_acquire", C.c_int32, [C.c_void_p, C.c_int32]),
    ("granikv_index_release", C.c_int32, [C.c_void_p, C.c_int32]),
    ("granikv_index_remove", C.c_int32, [C.c_void_p, C.c_int32]),
    ("granikv_index_info", C.c_int32, [C.c_void_p, C.c_int32, C.POINTER(PrefixInfo)]),
    ("granikv_index_stats", C.c_int32, [C.c_void_p, C.POINTER(C.c_int32), C.POINTER(C.c_int32),
                                        C.POINTER(C.c_int32)]),
    ("granikv_plan_create", C.c_int32, [C.c_void_p, C.POINTER(C.c_void_p)]),
    ("granikv_plan_destroy", C.c_int32, [C.c_void_p]),
    ("granikv_dispatch", C.c_int32, [C.c_void_p, C.POINTER(_Batch), C.c_void_p]),
    ("granikv_plan_num_groups", C.c_int32, [C.c_void_p, C.POINTER(C.c_int32)]),
    ("granikv_plan_group", C.c_int32, [C.c_void_p, C.c_int32, C.POINTER(GroupInfo)]),
    ("granikv_plan_schedule", C.c_int32, [C.c_void_p, C.POINTER(C.c_int32), C.POINTER(C.c_int32),
                                          C.POINTER(C.c_int32)]),
    ("granikv_workspace_size", C.c_int32, [C.c_void_p, C.c_void_p, C.POINTER(C.c_size_t)]),
    ("granikv_set_concurrency", C.c_int32, [C.c_void_p, C.c_int32, C.c_float]),
    ("granikv_set_fused_merge", C.c_int32, [C.c_void_p, C.c_int32]),
    ("granikv_set_dense_l2_ahead", C.c_int32, [C.c_void_p, C.c_int32]),
    ("granikv_plan_dense_l2_ahead", C.c_int32, [C.c_void_p, C.POINTER(C.c_int32)]),
    ("granikv_plan_suffix_runs", C.c_int32, [C.c_void_p, C.POINTER(C.c_int32), C.POINTER(C.c_int32)]),
    ("granikv_set_msat", C.c_int32, [C.c_void_p, C.c_int32]),
    ("granikv_get_msat", C.c_int32, [C.c_void_p, C.POINTER(C.c_int32)]),
    ("granikv_force_backend", C.c_int32, [C.c_void_p, C.c_int32]),
    ("granikv_decode_attention", C.c_int32, [C.c_void_p, C.c_int32, C.c_void_p, C.POINTER(_Batch),
                                             C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                             C.c_size_t, C.c_void_p]),
    ("granikv_decode_attention_append", C.c_int32, [C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p,
                                                    C.POINTER(_Batch), C.c_void_p, C.c_void_p, C.c_void_p,
                                                    C.c_void_p, C.c_size_t, C.c_void_p]),
    ("granikv_decode_attention_static", C.c_int32, [C.c_void_p, C.c_int32, C.c_void_p, C.POINTER(_Batch),
                                                    C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
    ("granikv_prefill_attention", C.c_int32, [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                                              C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t,
                                              C.c_void_p]),
    ("granikv_prefill_workspace_size", C.c_int32, [C.c_void_p, C.c_int32, C.POINTER(C.c_size_t)]),
    ("granikv_plan_image", C.c_int32, [C.c_void_p, C.c_void_p, C.c_size_t, C.POINTER(C.c_size_t)]),
    ("granikv_set_checks", C.c_int32, [C.c_void_p, C.c_int32]),
    ("granikv_inject_stall", C.c_int32, [C.c_void_p, C.c_int32]),
    ("granikv_sync_status", C.c_int32, [C.c_void_p, C.c_void_p]),
    ("granikv_launch_count", C.c_int32, [C.c_void_p, C.POINTER(C.c_int64), C.POINTER(C.c_int64)]),
]

EXPORTED = [s[0] for s in _SIGNATURES]


def load_library(path: Optional[str] = None):
    """Load libgranikv.so (once).  Raises RuntimeError if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"libgranikv.so is not built ({p} missing); build it with "
            "`python -m shared_prefix_kv_decode_gb300.build` (needs nvcc)")
    lib = C.CDLL(p)
    for name, res, args in _SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().granikv_status_string(status).decode()


def _check(status: int, where: str):
    if status == OK:
        return
    text = status_string(status)
    cls = {ERR_NO_HOT_SPACE: NoHotSpace, ERR_NO_COLD_SPACE: NoColdSpace,
           ERR_DEVICE_CHECK: DeviceCheckFailed}.get(status, GranikvError)
    raise cls(status, where, text)


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    raise TypeError(f"expected a device address or a tensor, got {type(x)}")


def _stream(s) -> Optional[int]:
    if s is None:
        return None
    if isinstance(s, int):
        return s or None
    if hasattr(s, "cuda_stream"):
        return int(s.cuda_stream) or None
    raise TypeError(f"expected a stream handle, got {type(s)}")


def _i32_array(values: Sequence[int]):
    arr = (C.c_int32 * len(values))(*[int(v) for v in values])
    return arr


class Batch:
    """Host-side batch descriptor (granikv_batch); keeps its host arrays alive."""

    def __init__(self, slab_id: Sequence[int], seq_len: Sequence[int], req_to_slot, cap: int, seq_len_dev=None):
        if len(slab_id) != len(seq_len):
            raise ValueError("slab_id and seq_len differ in length")
        self._slab = _i32_array(slab_id)
        self._len = _i32_array(seq_len)
        self._table = req_to_slot  # keep the tensors alive
        self._live = seq_len_dev
        self.c = _Batch(len(slab_id), C.cast(self._slab, C.POINTER(C.c_int32)),
                        C.cast(self._len, C.POINTER(C.c_int32)), _ptr(req_to_slot) or 0, int(cap),
                        _ptr(seq_len_dev))

    @property
    def B(self) -> int:
        return self.c.B


class Plan:
    def __init__(self, ctx: "Context"):
        self._ctx = ctx
        h = C.c_void_p()
        _check(ctx._lib.granikv_plan_create(ctx.handle, C.byref(h)), "granikv_plan_create")
        self.handle = h

    def groups(self):
        lib = self._ctx._lib
        n = C.c_int32()
        _check(lib.granikv_plan_num_groups(self.handle, C.byref(n)), "granikv_plan_num_groups")
        out = []
        for i in range(n.value):
            gi = GroupInfo()
            _check(lib.granikv_plan_group(self.handle, i, C.byref(gi)), "granikv_plan_group")
            out.append(gi.as_dict())
        return out

    def schedule(self) -> dict:
        """{"concurrent": bool, "prefix_ctas": int, "suffix_ctas": int} of the last dispatch."""
        a, b, c = C.c_int32(), C.c_int32(), C.c_int32()
        _check(self._ctx._lib.granikv_plan_schedule(self.handle, C.byref(a), C.byref(b), C.byref(c)),
               "granikv_plan_schedule")
        return {"concurrent": bool(a.value), "prefix_ctas": b.value, "suffix_ctas": c.value}

    def suffix_runs(self) -> dict:
        """{"runs": suffix runs (token-CTA work lists), "tail_runs": of them, those the one
        grid's dense CTAs take after their prefix piece}."""
        a, t = C.c_int32(), C.c_int32()
        _check(self._ctx._lib.granikv_plan_suffix_runs(self.handle, C.byref(a), C.byref(t)), "granikv_plan_suffix_runs")
        return {"runs": a.value, "tail_runs": t.value}

    def dense_l2_ahead(self) -> int:
        """Tiles the dense kernel reads ahead into L2 in this plan's launches (0: none)."""
        n = C.c_int32()
        _check(self._ctx._lib.granikv_plan_dense_l2_ahead(self.handle, C.byref(n)), "granikv_plan_dense_l2_ahead")
        return n.value

    def image(self) -> bytes:
        """The plan's device image (the work list copied into the workspace), for diagnostics."""
        lib = self._ctx._lib
        n = C.c_size_t()
        lib.granikv_plan_image(self.handle, None, 0, C.byref(n))
        buf = C.create_string_buffer(max(n.value, 1))
        _check(lib.granikv_plan_image(self.handle, buf, n.value, C.byref(n)), "granikv_plan_image")
        return buf.raw[:n.value]

    def close(self):
        if self.handle:
            self._ctx._lib.granikv_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Index:
    """A prefix index (granikv_index) over a context's HOT pool.  Methods follow the C entry
    points' names; prefixes are given as sequences of token ids."""

    def __init__(self, ctx: "Context"):
        self._ctx = ctx
        self._lib = ctx._lib
        h = C.c_void_p()
        _check(self._lib.granikv_index_create(ctx.handle, C.byref(h)), "granikv_index_create")
        self.handle = h
        ctx._indexes.append(weakref.ref(self))

    @staticmethod
    def _tokens(tokens: Sequence[int]):
        arr = _i32_array(tokens) if len(tokens) else (C.c_int32 * 1)()
        return arr, C.cast(arr, C.POINTER(C.c_int32)), len(tokens)

    def match(self, tokens: Sequence[int], acquire: bool = False) -> dict:
        arr, ptr, n = self._tokens(tokens)
        out = PrefixInfo()
        _check(self._lib.granikv_index_match(self.handle, ptr, n, 1 if acquire else 0, C.byref(out)),
               "granikv_index_match")
        return out.as_dict()

    def insert(self, tokens: Sequence[int], max_evicted: int = 1024):
        """Admit a prefix; returns (info dict, list of evicted prefix handles)."""
        arr, ptr, n = self._tokens(tokens)
        out = PrefixInfo()
        ev = (C.c_int32 * max(1, max_evicted))()
        n_ev = C.c_int32()
        _check(self._lib.granikv_index_insert(self.handle, ptr, n, C.byref(out),
                                              C.cast(ev, C.POINTER(C.c_int32)), max_evicted,
                                              C.byref(n_ev)), "granikv_index_insert")
        return out.as_dict(), [ev[i] for i in range(n_ev.value)]

    def acquire(self, prefix_id: int):
        _check(self._lib.granikv_index_acquire(self.handle, prefix_id), "granikv_index_acquire")

    def release(self, prefix_id: int):
        _check(self._lib.granikv_index_release(self.handle, prefix_id), "granikv_index_release")

    def remove(self, prefix_id: int):
        _check(self._lib.granikv_index_remove(self.handle, prefix_id), "granikv_index_remove")

    def info(self, prefix_id: int) -> dict:
        out = PrefixInfo()
        _check(self._lib.granikv_index_info(self.handle, prefix_id, C.byref(out)), "granikv_index_info")
        return out.as_dict()

    def stats(self):
        """(live prefixes, HOT prefixes, tree nodes)"""
        a, b, c = C.c_int32(), C.c_int32(), C.c_int32()
        _check(self._lib.granikv_index_stats(self.handle, C.byref(a), C.byref(b), C.byref(c)),
               "granikv_index_stats")
        return a.value, b.value, c.value

    def close(self):
        if getattr(self, "handle", None):
            self._lib.granikv_index_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Context:
    """A libgranikv context (granikv_ctx).  Methods follow the C entry points' names."""

    def __init__(self, *, n_layers: int, n_q: int, n_kv: int, head_dim: int, dtype: int,
                 n_slots: int, k_pools=(), v_pools=(), hot_fraction: float = 0.2,
                 cold_init_order: Optional[Sequence[int]] = None, m_sat: int = 0,
                 max_slabs: int = 0, max_batch: int = 0, device: int = 0, host_only: bool = False):
        self._lib = load_library()
        self._kp = (C.c_void_p * max(1, n_layers))(*[_ptr(p) for p in k_pools]) if k_pools else None
        self._vp = (C.c_void_p * max(1, n_layers))(*[_ptr(p) for p in v_pools]) if v_pools else None
        self._order = _i32_array(cold_init_order) if cold_init_order is not None else None
        cfg = _Config(n_layers, n_q, n_kv, head_dim, dtype, device, n_slots, hot_fraction,
                      C.cast(self._kp, C.POINTER(C.c_void_p)) if self._kp else None,
                      C.cast(self._vp, C.POINTER(C.c_void_p)) if self._vp else None,
                      C.cast(self._order, C.POINTER(C.c_int32)) if self._order else None,
                      m_sat, max_slabs, max_batch, 1 if host_only else 0)
        h = C.c_void_p()
        _check(self._lib.granikv_create(C.byref(cfg), C.byref(h)), "granikv_create")
        self.handle = h
        self.n_q, self.n_kv, self.head_dim, self.dtype = n_q, n_kv, head_dim, dtype
        self._indexes = []

    def index(self) -> Index:
        return Index(self)

    def close(self):
        if getattr(self, "handle", None):
            for ref in getattr(self, "_indexes", []):
                x = ref()
                if x is not None:
                    x.close()  # an index returns its slabs to this context's HOT pool
            self._lib.granikv_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # HOT pool
    def hot_alloc(self, L_p: int):
        sid, off = C.c_int32(), C.c_int64()
        _check(self._lib.granikv_hot_alloc(self.handle, L_p, C.byref(sid), C.byref(off)), "granikv_hot_alloc")
        return sid.value, off.value

    def hot_free(self, slab_id: int):
        _check(self._lib.granikv_hot_free(self.handle, slab_id), "granikv_hot_free")

    def hot_info(self, slab_id: int):
        off, L = C.c_int64(), C.c_int32()
        _check(self._lib.granikv_hot_info(self.handle, slab_id, C.byref(off), C.byref(L)), "granikv_hot_info")
        return off.value, L.value

    def hot_stats(self):
        n, m = C.c_int64(), C.c_int64()
        _check(self._lib.granikv_hot_stats(self.handle, C.byref(n), C.byref(m)), "granikv_hot_stats")
        return n.value, m.value

    def hot_fill(self, layer: int, slab_id: int, k, v, stream=None):
        _check(self._lib.granikv_hot_fill(self.handle, layer, slab_id, _ptr(k), _ptr(v), _stream(stream)),
               "granikv_hot_fill")

    # COLD pool
    def cold_alloc(self, n_new: Sequence[int], req_to_slot, suffix_len, cap: int, slots_out=None, stream=None):
        arr = _i32_array(n_new)
        _check(self._lib.granikv_cold_alloc(self.handle, C.cast(arr, C.POINTER(C.c_int32)), len(n_new),
                                            _ptr(req_to_slot), _ptr(suffix_len), cap, _ptr(slots_out),
                                            _stream(stream)), "granikv_cold_alloc")

    def cold_free(self, slots, n: int, stream=None):
        _check(self._lib.granikv_cold_free(self.handle, _ptr(slots), n, _stream(stream)), "granikv_cold_free")

    def cold_alloc_uniform(self, n: int, B: int, req_to_slot, suffix_len, cap: int, slots_out=None, stream=None):
        _check(self._lib.granikv_cold_alloc_uniform(self.handle, n, B, _ptr(req_to_slot), _ptr(suffix_len), cap,
                                                    _ptr(slots_out), _stream(stream)), "granikv_cold_alloc_uniform")

    def cold_sync(self, stream=None):
        _check(self._lib.granikv_cold_sync(self.handle, _stream(stream)), "granikv_cold_sync")

    def cold_free_count(self) -> int:
        n = C.c_int64()
        _check(self._lib.granikv_cold_free_count(self.handle, C.byref(n)), "granikv_cold_free_count")
        return n.value

    def cold_append(self, layer: int, k_new, v_new, slots, N: int, stream=None):
        _check(self._lib.granikv_cold_append(self.handle, layer, _ptr(k_new), _ptr(v_new), _ptr(slots), N,
                                             _stream(stream)), "granikv_cold_append")

    # dispatch
    def plan(self) -> Plan:
        return Plan(self)

    def dispatch(self, batch: Batch, plan: Optional[Plan] = None) -> Plan:
        plan = plan or Plan(self)
        _check(self._lib.granikv_dispatch(self.handle, C.byref(batch.c), plan.handle), "granikv_dispatch")
        return plan

    def workspace_size(self, plan: Plan) -> int:
        n = C.c_size_t()
        _check(self._lib.granikv_workspace_size(self.handle, plan.handle, C.byref(n)), "granikv_workspace_size")
        return n.value

    def set_concurrency(self, on: bool, prefix_sm_share: float = 0.0):
        _check(self._lib.granikv_set_concurrency(self.handle, 1 if on else 0, prefix_sm_share),
               "granikv_set_concurrency")

    def set_fused_merge(self, on: bool):
        _check(self._lib.granikv_set_fused_merge(self.handle, 1 if on else 0), "granikv_set_fused_merge")

    def set_dense_l2_ahead(self, tiles: int):
        """Dense kernel's L2 read-ahead in tiles: -1 automatic (the default), 0 off, 1-64 forced."""
        _check(self._lib.granikv_set_dense_l2_ahead(self.handle, int(tiles)), "granikv_set_dense_l2_ahead")

    def set_msat(self, m_sat: int):
        _check(self._lib.granikv_set_msat(self.handle, m_sat), "granikv_set_msat")

    def get_msat(self) -> int:
        m = C.c_int32()
        _check(self._lib.granikv_get_msat(self.handle, C.byref(m)), "granikv_get_msat")
        return m.value

    def force_backend(self, backend: int):
        _check(self._lib.granikv_force_backend(self.handle, backend), "granikv_force_backend")

    # decode attention
    def decode_attention(self, layer: int, q, batch: Batch, plan: Optional[Plan], o, lse, workspace,
                         ws_bytes: int, stream=None):
        _check(self._lib.granikv_decode_attention(self.handle, layer, _ptr(q), C.byref(batch.c),
                                                  plan.handle if plan is not None else None, _ptr(o),
                                                  _ptr(lse), _ptr(workspace), ws_bytes, _stream(stream)),
               "granikv_decode_attention")

    def decode_attention_append(self, layer: int, q, k_new, v_new, batch: Batch, plan: Optional[Plan], o, lse,
                                workspace, ws_bytes: int, stream=None):
        _check(self._lib.granikv_decode_attention_append(self.handle, layer, _ptr(q), _ptr(k_new), _ptr(v_new),
                                                         C.byref(batch.c), plan.handle if plan else None, _ptr(o),
                                                         _ptr(lse), _ptr(workspace), ws_bytes, _stream(stream)),
               "granikv_decode_attention_append")

    def decode_attention_static(self, layer: int, q, batch: Batch, plan: Plan, o, lse, stream=None):
        """Decode attention on the library's built-in workspace (no caller workspace, nothing
        allocated); see granikv_decode_attention_static in include/granikv.h."""
        _check(self._lib.granikv_decode_attention_static(self.handle, layer, _ptr(q), C.byref(batch.c),
                                                         plan.handle, _ptr(o), _ptr(lse), _stream(stream)),
               "granikv_decode_attention_static")

    # prefill of a HOT slab
    def prefill_workspace_size(self, L_p: int) -> int:
        n = C.c_size_t()
        _check(self._lib.granikv_prefill_workspace_size(self.handle, L_p, C.byref(n)),
               "granikv_prefill_workspace_size")
        return n.value

    def prefill_attention(self, layer: int, slab_id: int, k_new, v_new, q, o, lse, workspace, ws_bytes: int,
                          stream=None):
        _check(self._lib.granikv_prefill_attention(self.handle, layer, slab_id, _ptr(k_new), _ptr(v_new), _ptr(q),
                                                   _ptr(o), _ptr(lse), _ptr(workspace), ws_bytes, _stream(stream)),
               "granikv_prefill_attention")

    # checks
    def set_checks(self, on: bool):
        _check(self._lib.granikv_set_checks(self.handle, 1 if on else 0), "granikv_set_checks")

    def inject_stall(self, on: bool = True):
        """Test hook: the next decode call's first suffix token-CTA withholds its first tile (see
        granikv_inject_stall in include/granikv.h)."""
        _check(self._lib.granikv_inject_stall(self.handle, 1 if on else 0), "granikv_inject_stall")

    def sync_status(self, stream=None):
        _check(self._lib.granikv_sync_status(self.handle, _stream(stream)), "granikv_sync_status")

    def launch_count(self):
        k, c = C.c_int64(), C.c_int64()
        _check(self._lib.granikv_launch_count(self.handle, C.byref(k), C.byref(c)), "granikv_launch_count")
        return k.value, c.value

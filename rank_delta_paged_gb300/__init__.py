"""Python binding of libslora.so: the paged heterogeneous-rank LoRA delta on GB300.

Every function here has the name of the C entry point it calls (see ``include/slora.h``)
and only marshals arguments: device pointers, host pointers and sizes go through
``ctypes``; torch tensors and numpy arrays are accepted wherever the C call takes a
pointer and are passed as their data pointer.  No step of the hot path runs in Python
and there is no fallback: if ``libslora.so`` is missing, every call raises.

Build the library with ``rank_delta_paged_gb300.build.build()`` (nvcc, sm_103a).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

from . import build as _build

__all__ = [
    "SloraError", "lib", "library_path",
    "slora_status_str", "slora_last_error", "slora_version",
    "slora_pagealloc_create", "slora_pagealloc_destroy", "slora_pagealloc_alloc",
    "slora_pagealloc_free", "slora_pagealloc_num_free",
    "slora_pool_create", "slora_pool_destroy", "slora_pool_num_free", "slora_pool_base",
    "slora_pages_alloc", "slora_pages_free",
    "slora_adapter_register", "slora_adapter_unregister",
    "slora_adapter_load", "slora_adapters_load", "slora_adapter_evict", "slora_adapter_is_resident",
    "slora_lora_apply", "slora_lora_apply_noalloc",
    "slora_adapter_pages", "slora_adapter_rank", "slora_page_read", "slora_get_device_status",
    "slora_pool_launch_count",
    "slora_pool_set_stage_event",
    "slora_pool_set_load_mode", "slora_pool_get_load_mode", "slora_pool_set_load_start_event",
    "SLORA_LOAD_ZERO_COPY", "SLORA_LOAD_COPY_ENGINE",
    "slora_adapters_evict",
    "slora_debug_set_prefill_cluster",
    "slora_debug_set_prefill_split",
    "slora_debug_inject_load_fault", "SLORA_FAULT_NONE", "SLORA_FAULT_COPY", "SLORA_FAULT_SCATTER",
    "SLORA_FAULT_DIRECTORY", "SLORA_FAULT_STAGING", "SLORA_FAULT_ARENA",
    "slora_lora_apply_multi", "slora_plan_create", "slora_plan_apply", "slora_plan_remake",
    "slora_plan_destroy",
    "slora_lru_create", "slora_lru_destroy", "slora_lru_insert", "slora_lru_remove", "slora_lru_touch",
    "slora_lru_pin", "slora_lru_unpin", "slora_lru_victims",
    "slora_adapters_acquire", "slora_adapters_release", "slora_pages_alloc_evict", "slora_pool_get_stats",
    "slora_bmm_workspace_bytes", "slora_lora_apply_bmm",
]

_I32, _I64, _U64, _F32, _P = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p
_PP = ctypes.POINTER(ctypes.c_void_p)

# name -> argtypes (every function returns slora_status unless listed in _RESTYPE)
_SIGS = {
    "slora_status_str": [ctypes.c_int],
    "slora_last_error": [],
    "slora_version": [],
    "slora_pagealloc_create": [_I64, _U64, _PP],
    "slora_pagealloc_destroy": [_P],
    "slora_pagealloc_alloc": [_P, _I64, _P],
    "slora_pagealloc_free": [_P, _I64, _P],
    "slora_pagealloc_num_free": [_P, _P],
    "slora_pool_create": [ctypes.c_int, _I32, _I64, _I32, _I32, _U64, _PP],
    "slora_pool_destroy": [_P],
    "slora_pool_num_free": [_P, _P],
    "slora_pool_base": [_P, _PP],
    "slora_pages_alloc": [_P, _I64, _P],
    "slora_pages_free": [_P, _I64, _P, _P],
    "slora_adapter_register": [_P, _I32, _I32, _F32, _P, _P],
    "slora_adapter_unregister": [_P, _I32, _P],
    "slora_adapter_load": [_P, _I32, _P],
    "slora_adapters_load": [_P, _I32, _P, _P],
    "slora_adapter_evict": [_P, _I32, _P],
    "slora_adapter_is_resident": [_P, _I32, _P],
    "slora_lora_apply": [_P, _I32, _P, _P, _I32, _P, _P, _I32, _P, _P],
    "slora_lora_apply_noalloc": [_P, _I32, _P, _P, _I32, _P, _P, _I32, _P, _P],
    "slora_adapter_pages": [_P, _I32, _I32, _P],
    "slora_adapter_rank": [_P, _I32, _P],
    "slora_page_read": [_P, _I32, _P],
    "slora_get_device_status": [_P, _P],
    "slora_pool_launch_count": [_P, _P],
    "slora_pool_set_stage_event": [_P, _P],
    "slora_pool_set_load_mode": [_P, _I32, _I64],
    "slora_pool_get_load_mode": [_P, _P, _P],
    "slora_pool_set_load_start_event": [_P, _P],
    "slora_adapters_evict": [_P, _I32, _P, _P],
    "slora_debug_set_prefill_cluster": [_I32],
    "slora_debug_set_prefill_split": [_I32],
    "slora_debug_inject_load_fault": [_I32, _I32],
    "slora_lora_apply_multi": [_P, _I32, _P, _P, _P, _I32, _P, _P, _I32, _P, _P],
    "slora_plan_create": [_P, _I32, _I32, _P, _P, _I32, _P, _P, _PP],
    "slora_plan_apply": [_P, _I32, _P, _P, _P, _P],
    "slora_plan_remake": [_P, _P, _P, _P, _P],
    "slora_plan_destroy": [_P],
    "slora_lru_create": [_PP],
    "slora_lru_destroy": [_P],
    "slora_lru_insert": [_P, _I32],
    "slora_lru_remove": [_P, _I32],
    "slora_lru_touch": [_P, _I32],
    "slora_lru_pin": [_P, _I32],
    "slora_lru_unpin": [_P, _I32],
    "slora_lru_victims": [_P, _I32, _P, _I32, _P, _P],
    "slora_adapters_acquire": [_P, _I32, _P, _P],
    "slora_adapters_release": [_P, _I32, _P],
    "slora_pages_alloc_evict": [_P, _I64, _P, _P],
    "slora_pool_get_stats": [_P, _P],
    "slora_bmm_workspace_bytes": [_P, _I32, _P],
    "slora_lora_apply_bmm": [_P, _I32, _P, _P, _I32, _P, _P, _P, ctypes.c_size_t, _P],
}
_RESTYPE = {"slora_status_str": ctypes.c_char_p, "slora_last_error": ctypes.c_char_p,
            "slora_version": _I32}

_lock = threading.Lock()
_lib = None


class SloraError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} -> {msg}")
        self.status = status


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded libslora.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(f"libslora.so is not built ({path}); run "
                                   "rank_delta_paged_gb300.build.build() first")
            L = ctypes.CDLL(path)
            for name, args in _SIGS.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = _RESTYPE.get(name, ctypes.c_int)
            _lib = L
    return _lib


def _ptr(a) -> Optional[int]:
    """Data pointer of a torch tensor / numpy array / int / None."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if hasattr(a, "data_ptr"):
        return int(a.data_ptr())
    if hasattr(a, "ctypes"):
        return int(a.ctypes.data)
    raise TypeError(f"cannot take a pointer of {type(a)}")


def _stream(s) -> Optional[int]:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)  # torch.cuda.Stream


def _call(name: str, *args) -> None:
    st = getattr(lib(), name)(*args)
    if st != 0:
        raise SloraError(name, st, slora_last_error())


def slora_status_str(s: int) -> str:
    return lib().slora_status_str(int(s)).decode()


def slora_last_error() -> str:
    return lib().slora_last_error().decode()


def slora_version() -> int:
    return int(lib().slora_version())


# ---- host page allocator --------------------------------------------------------
def slora_pagealloc_create(num_pages: int, shuffle_seed: int = 0) -> int:
    h = ctypes.c_void_p()
    _call("slora_pagealloc_create", num_pages, shuffle_seed, ctypes.byref(h))
    return h.value


def slora_pagealloc_destroy(a: int) -> None:
    _call("slora_pagealloc_destroy", a)


def slora_pagealloc_alloc(a: int, n: int, out_pages) -> None:
    _call("slora_pagealloc_alloc", a, n, _ptr(out_pages))


def slora_pagealloc_free(a: int, n: int, pages) -> None:
    _call("slora_pagealloc_free", a, n, _ptr(pages))


def slora_pagealloc_num_free(a: int) -> int:
    v = ctypes.c_int64()
    _call("slora_pagealloc_num_free", a, ctypes.byref(v))
    return v.value


# ---- pool -------------------------------------------------------------------------
def slora_pool_create(device: int, hidden: int, num_pages: int, n_proj: int, max_adapters: int,
                      shuffle_seed: int = 0) -> int:
    h = ctypes.c_void_p()
    _call("slora_pool_create", device, hidden, num_pages, n_proj, max_adapters, shuffle_seed,
          ctypes.byref(h))
    return h.value


def slora_pool_destroy(pool: int) -> None:
    _call("slora_pool_destroy", pool)


def slora_pool_num_free(pool: int) -> int:
    v = ctypes.c_int64()
    _call("slora_pool_num_free", pool, ctypes.byref(v))
    return v.value


def slora_pool_base(pool: int) -> int:
    v = ctypes.c_void_p()
    _call("slora_pool_base", pool, ctypes.byref(v))
    return v.value


def slora_pages_alloc(pool: int, n: int, out_pages) -> None:
    _call("slora_pages_alloc", pool, n, _ptr(out_pages))


def slora_pages_free(pool: int, n: int, pages, stream=None) -> None:
    _call("slora_pages_free", pool, n, _ptr(pages), _stream(stream))


def slora_adapter_register(pool: int, adapter_id: int, rank: int, scaling: float, At_host,
                           B_host) -> None:
    _call("slora_adapter_register", pool, adapter_id, rank, scaling, _ptr(At_host), _ptr(B_host))


def slora_adapter_unregister(pool: int, adapter_id: int, stream=None) -> None:
    _call("slora_adapter_unregister", pool, adapter_id, _stream(stream))


def slora_adapter_load(pool: int, adapter_id: int, stream=None) -> None:
    _call("slora_adapter_load", pool, adapter_id, _stream(stream))


def slora_adapters_load(pool: int, n: int, adapter_ids, stream=None) -> None:
    _call("slora_adapters_load", pool, n, _ptr(adapter_ids), _stream(stream))


def slora_adapter_evict(pool: int, adapter_id: int, stream=None) -> None:
    _call("slora_adapter_evict", pool, adapter_id, _stream(stream))


def slora_adapters_evict(pool: int, n: int, adapter_ids, stream=None) -> None:
    _call("slora_adapters_evict", pool, n, _ptr(adapter_ids), _stream(stream))


def slora_adapter_is_resident(pool: int, adapter_id: int) -> bool:
    v = ctypes.c_int32()
    _call("slora_adapter_is_resident", pool, adapter_id, ctypes.byref(v))
    return bool(v.value)


def slora_lora_apply(pool: int, proj: int, x, y, T: int, token_adapter_idx, seg_indptr=None,
                     n_seg: int = 0, scaling=None, stream=None) -> None:
    _call("slora_lora_apply", pool, proj, _ptr(x), _ptr(y), T, _ptr(token_adapter_idx),
          _ptr(seg_indptr), n_seg, _ptr(scaling), _stream(stream))


def slora_lora_apply_noalloc(pool: int, proj: int, x, y, T: int, token_adapter_idx,
                             seg_indptr=None, n_seg: int = 0, scaling=None, stream=None) -> None:
    """slora_lora_apply without device allocation: plan scratch in the library's fixed
    device array (see include/slora.h for the size limit and the sharing rules)."""
    _call("slora_lora_apply_noalloc", pool, proj, _ptr(x), _ptr(y), T, _ptr(token_adapter_idx),
          _ptr(seg_indptr), n_seg, _ptr(scaling), _stream(stream))


def slora_lora_apply_multi(pool: int, projs, xs, ys, T: int, token_adapter_idx, seg_indptr=None,
                           n_seg: int = 0, scaling=None, stream=None) -> None:
    """One call for several projections of a layer: projs[j], xs[j], ys[j] per entry (the
    host arrays of projection indices and device pointers are built here)."""
    n = len(projs)
    if len(xs) != n or len(ys) != n:
        raise ValueError("projs, xs and ys must have the same length")
    p_arr = (ctypes.c_int32 * max(n, 1))(*[int(v) for v in projs])
    x_arr = (ctypes.c_void_p * max(n, 1))(*[_ptr(v) for v in xs])
    y_arr = (ctypes.c_void_p * max(n, 1))(*[_ptr(v) for v in ys])
    _call("slora_lora_apply_multi", pool, n, p_arr, x_arr, y_arr, T, _ptr(token_adapter_idx),
          _ptr(seg_indptr), n_seg, _ptr(scaling), _stream(stream))


def slora_plan_create(pool: int, n_slots: int, T: int, token_adapter_idx, seg_indptr=None, n_seg: int = 0,
                      scaling=None, stream=None) -> int:
    """The plan of a batch for n_slots projections per apply, made once for the layers of an
    iteration; returns the plan handle."""
    out = ctypes.c_void_p()
    _call("slora_plan_create", pool, n_slots, T, _ptr(token_adapter_idx), _ptr(seg_indptr), n_seg,
          _ptr(scaling), _stream(stream), ctypes.byref(out))
    return int(out.value)


def slora_plan_apply(plan: int, projs, xs, ys, stream=None) -> None:
    """One layer of a planned batch: projs[j], xs[j], ys[j] per projection slot."""
    n = len(projs)
    if len(xs) != n or len(ys) != n:
        raise ValueError("projs, xs and ys must have the same length")
    p_arr = (ctypes.c_int32 * max(n, 1))(*[int(v) for v in projs])
    x_arr = (ctypes.c_void_p * max(n, 1))(*[_ptr(v) for v in xs])
    y_arr = (ctypes.c_void_p * max(n, 1))(*[_ptr(v) for v in ys])
    _call("slora_plan_apply", plan, n, p_arr, x_arr, y_arr, _stream(stream))


def slora_plan_remake(plan: int, token_adapter_idx, seg_indptr=None, scaling=None, stream=None) -> None:
    """The next batch (same T, n_seg and projections per apply) planned into the same plan."""
    _call("slora_plan_remake", plan, _ptr(token_adapter_idx), _ptr(seg_indptr), _ptr(scaling), _stream(stream))


def slora_plan_destroy(plan: int) -> None:
    _call("slora_plan_destroy", plan)


# ---- recency index (host only) and residency under pressure ------------------------
class PoolStats(ctypes.Structure):
    _fields_ = [("free_pages", ctypes.c_int64), ("resident_adapters", ctypes.c_int64),
                ("pinned_adapters", ctypes.c_int64), ("adapters_loaded", ctypes.c_int64),
                ("adapters_evicted", ctypes.c_int64)]

    def as_dict(self) -> dict:
        return {f: int(getattr(self, f)) for f, _ in self._fields_}


def _ids(ids):
    import numpy as np
    a = np.ascontiguousarray(np.asarray(list(ids) if not hasattr(ids, "dtype") else ids, dtype=np.int32))
    return a, int(a.shape[0])


def slora_lru_create() -> int:
    h = ctypes.c_void_p()
    _call("slora_lru_create", ctypes.byref(h))
    return h.value


def slora_lru_destroy(lru: int) -> None:
    _call("slora_lru_destroy", lru)


def slora_lru_insert(lru: int, adapter_id: int) -> None:
    _call("slora_lru_insert", lru, adapter_id)


def slora_lru_remove(lru: int, adapter_id: int) -> None:
    _call("slora_lru_remove", lru, adapter_id)


def slora_lru_touch(lru: int, adapter_id: int) -> None:
    _call("slora_lru_touch", lru, adapter_id)


def slora_lru_pin(lru: int, adapter_id: int) -> None:
    _call("slora_lru_pin", lru, adapter_id)


def slora_lru_unpin(lru: int, adapter_id: int) -> None:
    _call("slora_lru_unpin", lru, adapter_id)


def slora_lru_victims(lru: int, exclude=(), max_out: int = 1 << 20) -> list:
    """Up to max_out unpinned ids not in exclude, least recently used first."""
    import numpy as np
    ex, n_ex = _ids(exclude)
    n_all = ctypes.c_int32()
    out = np.empty(max(1, min(max_out, 1 << 20)), np.int32)
    _call("slora_lru_victims", lru, n_ex, ex.ctypes.data if n_ex else None, int(out.shape[0]),
          out.ctypes.data, ctypes.byref(n_all))
    return out[:n_all.value].tolist()


def slora_adapters_acquire(pool: int, adapter_ids, stream=None) -> None:
    a, n = _ids(adapter_ids)
    _call("slora_adapters_acquire", pool, n, a.ctypes.data if n else None, _stream(stream))


def slora_adapters_release(pool: int, adapter_ids) -> None:
    a, n = _ids(adapter_ids)
    _call("slora_adapters_release", pool, n, a.ctypes.data if n else None)


def slora_pages_alloc_evict(pool: int, n: int, out_pages, stream=None) -> None:
    _call("slora_pages_alloc_evict", pool, n, _ptr(out_pages), _stream(stream))


def slora_pool_get_stats(pool: int) -> dict:
    st = PoolStats()
    _call("slora_pool_get_stats", pool, ctypes.byref(st))
    return st.as_dict()


def slora_bmm_workspace_bytes(pool: int, T: int) -> int:
    v = ctypes.c_size_t()
    _call("slora_bmm_workspace_bytes", pool, T, ctypes.byref(v))
    return v.value


def slora_lora_apply_bmm(pool: int, proj: int, x, y, T: int, token_adapter_idx, workspace, workspace_bytes: int,
                         scaling=None, stream=None) -> None:
    """The padded batched-GEMM comparison path (see include/slora.h)."""
    _call("slora_lora_apply_bmm", pool, proj, _ptr(x), _ptr(y), T, _ptr(token_adapter_idx), _ptr(scaling),
          _ptr(workspace), int(workspace_bytes), _stream(stream))


def slora_adapter_pages(pool: int, adapter_id: int, proj: int, out) -> None:
    _call("slora_adapter_pages", pool, adapter_id, proj, _ptr(out))


def slora_adapter_rank(pool: int, adapter_id: int) -> int:
    v = ctypes.c_int32()
    _call("slora_adapter_rank", pool, adapter_id, ctypes.byref(v))
    return v.value


def slora_page_read(pool: int, page: int, host_out) -> None:
    _call("slora_page_read", pool, page, _ptr(host_out))


def slora_get_device_status(pool: int) -> int:
    v = ctypes.c_int32()
    _call("slora_get_device_status", pool, ctypes.byref(v))
    return v.value


def slora_pool_launch_count(pool: int) -> int:
    v = ctypes.c_int64()
    _call("slora_pool_launch_count", pool, ctypes.byref(v))
    return v.value


SLORA_FAULT_NONE, SLORA_FAULT_COPY, SLORA_FAULT_SCATTER = 0, 1, 2
SLORA_FAULT_DIRECTORY, SLORA_FAULT_STAGING, SLORA_FAULT_ARENA = 3, 4, 5


def slora_debug_inject_load_fault(kind: int, nth: int) -> None:
    """Make the nth later load-path operation of `kind` fail on the host (test hook)."""
    _call("slora_debug_inject_load_fault", int(kind), int(nth))


def slora_debug_set_prefill_cluster(ctas: int) -> None:
    """Force the prefill kernel's CTAs per cluster (1, 2, 4, 8) for later calls; 0 = auto."""
    _call("slora_debug_set_prefill_cluster", int(ctas))


def slora_debug_set_prefill_split(on: int) -> None:
    """Allow (1, the default) or forbid (0) splitting prefill units by expand columns."""
    _call("slora_debug_set_prefill_split", int(on))


SLORA_LOAD_ZERO_COPY = 0
SLORA_LOAD_COPY_ENGINE = 1


def slora_pool_set_load_mode(pool: int, mode: int, staging_bytes: int = 0) -> None:
    """Choose the load path: SLORA_LOAD_ZERO_COPY or SLORA_LOAD_COPY_ENGINE (staging ring of
    ``staging_bytes``, 0 = the library's default)."""
    _call("slora_pool_set_load_mode", pool, int(mode), int(staging_bytes))


def slora_pool_get_load_mode(pool: int):
    """(mode, staging_bytes) of the pool's load path."""
    m, b = ctypes.c_int32(), ctypes.c_int64()
    _call("slora_pool_get_load_mode", pool, ctypes.byref(m), ctypes.byref(b))
    return m.value, b.value


def slora_pool_set_load_start_event(pool: int, event) -> None:
    """Record `event` (a torch.cuda.Event, a raw cudaEvent_t as int, or None) on the pool's
    side stream before the work of every later load; None clears it."""
    handle = 0 if event is None else int(getattr(event, "cuda_event", event))
    _call("slora_pool_set_load_start_event", pool, ctypes.c_void_p(handle))


def slora_pool_set_stage_event(pool: int, event) -> None:
    """Record `event` (a torch.cuda.Event, a raw cudaEvent_t as int, or None) between the
    plan and the delta kernels of every apply of the pool; None clears it."""
    handle = 0 if event is None else int(getattr(event, "cuda_event", event))
    _call("slora_pool_set_stage_event", pool, ctypes.c_void_p(handle))

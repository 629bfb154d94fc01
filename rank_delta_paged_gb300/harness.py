"""Set up a pool for a seeded workload through the C ABI (orchestration only).

``PoolSession`` creates a pool shaped for a ``workloads.Workload``, takes the workload's
KV share of the slots through the shared free list, registers adapters in the pinned
host store, loads them, and calls the hot path.  Device tensors come from PyTorch (the
allocator and streams); every computation runs in libslora.so.
"""
from __future__ import annotations

from typing import Iterable, Optional

import numpy as np
import torch

from . import (slora_adapter_register, slora_adapters_load, slora_adapters_evict,
               slora_get_device_status, slora_lora_apply, slora_pages_alloc, slora_pool_create,
               slora_pool_destroy, slora_adapter_is_resident)
from .workloads import Workload


class PoolSession:
    def __init__(self, w: Workload, device: int = 0, max_adapters: Optional[int] = None):
        self.w = w
        self.device = device
        self.pool = slora_pool_create(device, w.hidden, w.num_pages, w.n_proj,
                                      max_adapters or w.n_adapters, w.shuffle_seed)
        self.kv_pages = np.empty(w.kv_pages, dtype=np.int32)
        if w.kv_pages:
            slora_pages_alloc(self.pool, w.kv_pages, self.kv_pages)
        self.registered = set()

    # ---- host store / residency -------------------------------------------------
    def register(self, ids: Iterable[int]) -> None:
        todo = [int(a) for a in ids if int(a) not in self.registered]
        self.w.prefetch_factors(todo)
        for a in todo:
            At, B = self.w.factors(a)
            slora_adapter_register(self.pool, a, int(self.w.ranks[a]), float(self.w.scaling()[a]),
                                   At, B)
            self.registered.add(a)

    def load(self, ids: Iterable[int], stream=None) -> None:
        ids = np.ascontiguousarray(np.asarray(list(ids), dtype=np.int32))
        self.register(ids.tolist())
        slora_adapters_load(self.pool, int(ids.shape[0]), ids, stream)

    def evict(self, ids: Iterable[int], stream=None) -> None:
        ids = np.ascontiguousarray(np.asarray(list(ids), dtype=np.int32))
        slora_adapters_evict(self.pool, int(ids.shape[0]), ids, stream)

    # ---- device inputs ------------------------------------------------------------
    def device_inputs(self, p: int = 0):
        """(x, y0, idx, seg_indptr) for projection p as device tensors."""
        dev = torch.device("cuda", self.device)
        x = torch.from_numpy(self.w.x(p).view(np.int16)).to(dev).view(torch.float16)
        y0 = torch.from_numpy(self.w.y0(p).view(np.int16)).to(dev).view(torch.float16)
        idx = torch.from_numpy(self.w.token_adapter_idx).to(dev)
        seg = None if self.w.seg_indptr is None else torch.from_numpy(self.w.seg_indptr).to(dev)
        return x, y0, idx, seg

    def apply(self, p: int, x, y, idx, seg=None, scaling=None, stream=None) -> None:
        n_seg = 0 if seg is None else int(seg.numel() - 1)
        slora_lora_apply(self.pool, p, x, y, int(idx.numel()), idx, seg, n_seg, scaling, stream)

    def device_status(self) -> int:
        return slora_get_device_status(self.pool)

    def close(self) -> None:
        if self.pool:
            slora_pool_destroy(self.pool)
            self.pool = 0

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def prefetch_overlap(sess: PoolSession, K: int = 6, stream=None, mode: Optional[int] = None) -> dict:
    """How far the adapter loads of later batches hide behind the deltas of earlier ones.

    The pool runs every load on its own side stream and only makes the caller's stream
    wait for it, so a serving loop that issues load(k), apply(k), load(k+1), apply(k+1), ...
    on one stream already lets load(k+1) run under apply(k) (S-LoRA: Serving Thousands of
    Concurrent LoRA Adapters (explainer), "Algorithm / figure walkthrough" step 2: the
    factors of the next iteration's adapters are prefetched into the pool while the current
    one computes).  K decode batches are drawn from the
    session's zoo (``Workload.later_batch``), starting from an empty pool; each loads the
    adapters not yet resident.  Timed on the stream with CUDA events:

      loads_ms       the K loads alone
      applies_ms     the K applies alone (every adapter resident)
      pipelined_ms   load(k), apply(k) in turn on one stream
      serialized_ms  the same with the host waiting for the device after every apply, so no
                     load starts before the previous apply ends
      overlap_frac   (loads + applies - pipelined) / min(loads, applies)
      link_gb_per_s  loaded bytes / loads_ms

    ``mode`` selects the pool's load path first (SLORA_LOAD_ZERO_COPY: the load kernel reads
    the pinned store over the CPU-GPU link; SLORA_LOAD_COPY_ENGINE: cudaMemcpyAsync into a
    staging ring, then the load kernel from HBM); None keeps the pool's current one.
    """
    from . import slora_lora_apply, slora_pool_get_load_mode, slora_pool_set_load_mode
    if mode is not None:
        slora_pool_set_load_mode(sess.pool, mode)
    w = sess.w
    batches = [w] + [w.later_batch(k) for k in range(1, K)]
    dev = torch.device("cuda", sess.device)
    st = stream or torch.cuda.current_stream(dev)
    x = [torch.from_numpy(w.x(p).view(np.int16)).to(dev).view(torch.float16) for p in range(w.n_proj)]
    y = [torch.from_numpy(w.y0(p).view(np.int16)).to(dev).view(torch.float16) for p in range(w.n_proj)]
    idx = [torch.from_numpy(b.token_adapter_idx).to(dev) for b in batches]
    need, resident = [], set()
    for b in batches:
        ids = [a for a in b.used_adapters().tolist() if a not in resident]
        need.append(ids)
        resident |= set(ids)
    union = sorted(resident)
    sess.register(union)
    nbytes = sum(4 * int(w.ranks[a]) * w.hidden * w.n_proj for ids in need for a in ids)

    def evict_all():
        res = [a for a in union if slora_adapter_is_resident(sess.pool, a)]
        if res:
            sess.evict(res, st)
        torch.cuda.synchronize(dev)

    def apply(k):
        for p in range(w.n_proj):
            slora_lora_apply(sess.pool, p, x[p], y[p], w.T, idx[k], None, 0, None, st)

    def timed(mode):
        if mode == "applies":
            sess.load(union, st)
        else:
            evict_all()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for k in range(K):
            if mode != "applies" and need[k]:
                sess.load(need[k], st)
            if mode != "loads":
                apply(k)
            if mode == "serialized":
                torch.cuda.synchronize(dev)
        e1.record(st)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    best = {}
    for _ in range(2):   # the faster of two passes of each
        for mode in ("loads", "applies", "pipelined", "serialized"):
            t = timed(mode)
            best[mode] = min(best.get(mode, t), t)
    evict_all()
    loads, applies, pipe = best["loads"], best["applies"], best["pipelined"]
    return {"load_mode": ["zero_copy", "copy_engine"][slora_pool_get_load_mode(sess.pool)[0]],
            "batches": K, "adapters_loaded": len(union), "bytes": int(nbytes),
            "loads_ms": loads, "applies_ms": applies, "pipelined_ms": pipe,
            "serialized_ms": best["serialized"],
            "overlap_frac": (loads + applies - pipe) / max(1e-9, min(loads, applies)),
            "link_gb_per_s": nbytes / (loads * 1e-3) / 1e9}


def pressure_run(sess: PoolSession, K: int = 6, stream=None) -> dict:
    """K batches from the session's zoo through a pool too small to keep them all: per
    batch, acquire its adapters (the pool evicts the least recently used ones that no batch
    holds), apply every layer (one slora_lora_apply_multi call per layer), release.

    Returns per-batch adapters used / already resident / loaded / evicted, the host time of
    the acquire call, and the device time from the acquire's first enqueued work to the
    end of the batch's last layer (CUDA events on the stream).  The explainer's "The
    mechanism": adapters that the running batches do not use leave GPU memory and stay in
    host memory; KV and adapters compete for one pool.
    """
    import time
    from . import (slora_adapters_acquire, slora_adapters_release, slora_lora_apply_multi,
                   slora_pool_get_stats)
    w = sess.w
    batches = [w] + [w.later_batch(k) for k in range(1, K)]
    dev = torch.device("cuda", sess.device)
    st = stream or torch.cuda.current_stream(dev)
    per_layer = w.n_proj // w.n_layers
    x = [torch.from_numpy(w.x(p).view(np.int16)).to(dev).view(torch.float16) for p in range(w.n_proj)]
    y = [torch.from_numpy(w.y0(p).view(np.int16)).to(dev).view(torch.float16) for p in range(w.n_proj)]
    seg = None if w.seg_indptr is None else torch.from_numpy(w.seg_indptr).to(dev)
    n_seg = w.n_seg
    sess.register(sorted(set().union(*[set(b.used_adapters().tolist()) for b in batches])))
    rows = []
    for b in batches:
        used = b.used_adapters()
        idx = torch.from_numpy(b.token_adapter_idx).to(dev)
        before = slora_pool_get_stats(sess.pool)
        was = sum(1 for a in used.tolist() if slora_adapter_is_resident(sess.pool, a))
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        t0 = time.perf_counter()
        slora_adapters_acquire(sess.pool, used, st)
        host_ms = 1e3 * (time.perf_counter() - t0)
        for l in range(w.n_layers):
            ps = list(range(l * per_layer, (l + 1) * per_layer))
            slora_lora_apply_multi(sess.pool, ps, [x[p] for p in ps], [y[p] for p in ps], b.T, idx, seg, n_seg,
                                   None, st)
        slora_adapters_release(sess.pool, used)
        e1.record(st)
        torch.cuda.synchronize(dev)
        after = slora_pool_get_stats(sess.pool)
        rows.append({"used": int(used.size), "resident_before": was,
                     "loaded": after["adapters_loaded"] - before["adapters_loaded"],
                     "evicted": after["adapters_evicted"] - before["adapters_evicted"],
                     "acquire_host_ms": host_ms, "device_ms": e0.elapsed_time(e1)})
    used = sum(r["used"] for r in rows[1:])
    return {"batches": K, "pool_adapter_pages": int(w.num_pages - w.kv_pages),
            "per_batch": rows,
            "hit_rate_after_first": (sum(r["resident_before"] for r in rows[1:]) / used) if used else None}

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

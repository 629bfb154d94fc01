"""CPU checks of host-side logic that the measurements rest on: the byte and flop counts
bench.py divides by, and the later batches the prefetch / pressure runs draw.  No GPU."""
import importlib.util
import os

import numpy as np

from rank_delta_paged_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_algorithmic_bytes_and_flops_by_hand():
    # hidden 64, two projections; adapters of rank 8 and 16 used, one base-only token
    w = W.Workload("hand", 64, 2, np.array([8, 16, 32], np.int32), np.array([0, 0, 1, -1], np.int32), None,
                   num_pages=64, kv_pages=0, shuffle_seed=0)
    b = _bench()
    # per projection: A^T and B rows of adapters 0 and 1 once (4 * r * d bytes each), x and
    # y0 read and y written for all 4 tokens (6 * d * T bytes)
    per_proj = 4 * 8 * 64 + 4 * 16 * 64 + 6 * 64 * 4
    assert b.algorithmic_bytes(w) == 2 * per_proj
    # 4 * d * r flops per token with an adapter (shrink and expand, multiply-add = 2)
    assert b.algorithmic_flops(w) == 2 * 4 * 64 * (8 + 8 + 16)


def test_later_batches_keep_the_zoo_and_the_shape():
    w = W.mixed_iteration(n_layers=1, n_adapters=50, pool_bytes=64 << 20)
    for k in (1, 2):
        b = w.later_batch(k)
        assert b.T == w.T and np.array_equal(b.seg_indptr, w.seg_indptr)
        assert np.array_equal(b.ranks, w.ranks) and b.seed == w.seed and b.num_pages == w.num_pages
        ids = b.token_adapter_idx
        assert ids.min() >= 0 and ids.max() < w.n_adapters
        for i in range(b.n_seg):   # one adapter per prefill request
            assert np.unique(ids[b.seg_indptr[i]:b.seg_indptr[i + 1]]).size == 1
        assert np.array_equal(ids, w.later_batch(k).token_adapter_idx)   # seeded
    assert not np.array_equal(w.later_batch(1).token_adapter_idx, w.later_batch(2).token_adapter_idx)
    d = W.decode_7b(T=64)
    nb = d.later_batch(3)
    assert nb.seg_indptr is None and nb.T == 64 and nb.alpha == d.alpha
    # the factors of an adapter are the same in every later batch (same zoo)
    a = int(nb.used_adapters()[0])
    assert all(np.array_equal(x, y) for x, y in zip(d.factors(a, cache=False), nb.factors(a, cache=False)))

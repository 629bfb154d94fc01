"""GPU checks of residency under pool pressure: slora_adapters_acquire / release evict the
least recently used adapters that no batch holds, slora_pages_alloc_evict lets KV blocks
grow into the adapters' share, held adapters never leave, a request that cannot fit
changes nothing, and the delta stays exact across eviction / reload cycles (pages
relocated)."""
import numpy as np
import pytest
import torch

import oracle
import rank_delta_paged_gb300 as rdp
from rank_delta_paged_gb300 import workloads as W
from rank_delta_paged_gb300.harness import PoolSession

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rdp.build.build()
    rdp.lib()


def small_pool(n_adapters=10, slots=5, kv=16):
    """Rank-8 adapters at hidden 256 (16 pages each) in a pool with room for `slots`."""
    ranks = np.full(n_adapters, 8, np.int32)
    idx = np.arange(n_adapters, dtype=np.int32)
    w = W.Workload("residency", 256, 1, ranks, idx, None, num_pages=16 * slots + kv, kv_pages=kv,
                   shuffle_seed=3, seed=1)
    s = PoolSession(w)
    s.register(range(n_adapters))
    return w, s


def resident(s, ids):
    return {a for a in ids if rdp.slora_adapter_is_resident(s.pool, a)}


def test_acquire_evicts_least_recently_used_unheld_adapters():
    w, s = small_pool()
    with s:
        acq, rel = rdp.slora_adapters_acquire, rdp.slora_adapters_release
        acq(s.pool, [0, 1, 2]); rel(s.pool, [0, 1, 2])
        acq(s.pool, [3, 4]); rel(s.pool, [3, 4])
        acq(s.pool, [0]); rel(s.pool, [0])                # 0 becomes the most recent
        assert rdp.slora_pool_get_stats(s.pool)["free_pages"] == 0
        acq(s.pool, [5, 6]); rel(s.pool, [5, 6])          # evicts 1 and 2
        assert resident(s, range(10)) == {0, 3, 4, 5, 6}
        acq(s.pool, [3])                                  # held from here on
        acq(s.pool, [7, 8, 9]); rel(s.pool, [7, 8, 9])    # evicts 4, 0, 5; never 3
        assert resident(s, range(10)) == {3, 6, 7, 8, 9}
        st = rdp.slora_pool_get_stats(s.pool)
        assert (st["adapters_loaded"], st["adapters_evicted"], st["pinned_adapters"]) == (10, 5, 1)
        # five adapters cannot fit beside the held one: nothing changes
        with pytest.raises(rdp.SloraError) as ei:
            acq(s.pool, [0, 1, 2, 4, 5])
        assert ei.value.status == 2                       # SLORA_ERR_POOL_FULL
        assert resident(s, range(10)) == {3, 6, 7, 8, 9}
        assert rdp.slora_pool_get_stats(s.pool) == st
        # a held adapter cannot be evicted by hand; release needs a hold
        with pytest.raises(rdp.SloraError):
            rdp.slora_adapter_evict(s.pool, 3)
        with pytest.raises(rdp.SloraError):
            rdp.slora_adapters_evict(s.pool, 2, np.array([6, 3], np.int32))
        assert resident(s, range(10)) == {3, 6, 7, 8, 9}
        rel(s.pool, [3])
        with pytest.raises(rdp.SloraError):
            rel(s.pool, [3])
        rdp.slora_adapter_evict(s.pool, 3)
        torch.cuda.synchronize()
        assert s.device_status() == 0


def test_kv_pages_grow_into_unheld_adapters():
    w, s = small_pool()
    with s:
        for a in range(5):
            rdp.slora_adapters_acquire(s.pool, [a])
            rdp.slora_adapters_release(s.pool, [a])
        rdp.slora_adapters_acquire(s.pool, [1])           # held
        pages = np.empty(40, np.int32)
        rdp.slora_pages_alloc_evict(s.pool, 40, pages)    # 40 pages: evicts 0, 2, 3 (48 pages)
        assert resident(s, range(5)) == {1, 4}
        assert rdp.slora_pool_get_stats(s.pool)["free_pages"] == 8
        assert len(set(pages.tolist())) == 40
        more = np.empty(40, np.int32)
        with pytest.raises(rdp.SloraError) as ei:         # only 4 (16 pages) can still go
            rdp.slora_pages_alloc_evict(s.pool, 40, more)
        assert ei.value.status == 2
        assert resident(s, range(5)) == {1, 4}
        rdp.slora_pages_free(s.pool, 40, pages)
        rdp.slora_adapters_release(s.pool, [1])
        torch.cuda.synchronize()


def test_exact_results_through_eviction_and_reload_cycles():
    """Decode batches from one zoo through a pool that holds about half of it: each batch
    acquires its adapters (evicting others, reloading earlier ones into other pages),
    applies, releases; every batch equals the oracle bit for bit."""
    ranks = np.array([[8, 16, 24, 32, 40, 48, 56, 64][i % 8] for i in range(40)], np.int32)
    base = W.Workload("churn", 512, 2, ranks, np.zeros(12, np.int32), None, num_pages=1, kv_pages=0,
                      shuffle_seed=5, seed=9, values="exact", alpha=0.8)
    batches = [base.later_batch(k) for k in range(8)]
    need = max(sum(2 * int(ranks[a]) * 2 for a in b.used_adapters()) for b in batches)
    num_pages = need + 256 + 64   # room for the largest batch and a little more
    w = W.Workload("churn", 512, 2, ranks, base.token_adapter_idx, None, num_pages=num_pages, kv_pages=64,
                   shuffle_seed=5, seed=9, values="exact", alpha=0.8)
    with PoolSession(w) as s:
        s.register(range(len(ranks)))
        dev = torch.device("cuda")
        for k, b in enumerate(batches):
            ids = b.used_adapters()
            rdp.slora_adapters_acquire(s.pool, ids)
            idx = torch.from_numpy(b.token_adapter_idx).to(dev)
            for p in range(2):
                x = torch.from_numpy(b.x(p).view(np.int16)).to(dev).view(torch.float16)
                y = torch.from_numpy(b.y0(p).view(np.int16)).to(dev).view(torch.float16)
                rdp.slora_lora_apply(s.pool, p, x, y, b.T, idx)
                torch.cuda.synchronize()
                got = y.cpu().view(torch.int16).numpy().view(np.uint16)
                ref = oracle.workload_reference(b, p=p).astype(np.float16).view(np.uint16)
                assert np.array_equal(got, ref), (k, p)
            rdp.slora_adapters_release(s.pool, ids)
        st = rdp.slora_pool_get_stats(s.pool)
        assert st["adapters_evicted"] > 0 and st["pinned_adapters"] == 0
        assert s.device_status() == 0

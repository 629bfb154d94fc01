"""CPU-side checks of the C ABI: the library builds for sm_103a, loads, exports every
entry point include/slora.h declares, and its host page allocator (the free list the
pool shares between adapter rows and KV blocks) behaves as documented.  No GPU calls."""
import ctypes
import os
import re
import shutil

import numpy as np
import pytest

import rank_delta_paged_gb300 as rdp
from rank_delta_paged_gb300 import build as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "slora.h")

pytestmark = pytest.mark.skipif(shutil.which(B.NVCC) is None, reason="nvcc not available")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return rdp.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(slora_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for must in ("slora_pool_create", "slora_adapter_load", "slora_adapter_evict",
                 "slora_lora_apply", "slora_pages_alloc", "slora_adapter_register"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding wraps each of them under the same name
    unwrapped = [n for n in declared_functions() if not hasattr(rdp, n)]
    assert not unwrapped, unwrapped


def test_status_strings(lib):
    assert rdp.slora_status_str(0) == "SLORA_OK"
    assert rdp.slora_status_str(2) == "SLORA_ERR_POOL_FULL"
    assert rdp.slora_version() >= 100


def test_library_targets_sm103a():
    # the objects were built with the sm_103a gencode only
    assert B.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_pagealloc_unshuffled_order(lib):
    a = rdp.slora_pagealloc_create(16, 0)
    try:
        out = np.empty(5, np.int32)
        rdp.slora_pagealloc_alloc(a, 5, out)
        assert out.tolist() == [0, 1, 2, 3, 4]
        assert rdp.slora_pagealloc_num_free(a) == 11
    finally:
        rdp.slora_pagealloc_destroy(a)


def test_pagealloc_shuffle_is_seeded_permutation(lib):
    def draw(seed):
        a = rdp.slora_pagealloc_create(1000, seed)
        out = np.empty(1000, np.int32)
        rdp.slora_pagealloc_alloc(a, 1000, out)
        rdp.slora_pagealloc_destroy(a)
        return out
    x, y, z = draw(7), draw(7), draw(8)
    assert np.array_equal(np.sort(x), np.arange(1000))      # a permutation
    assert np.array_equal(x, y)                              # deterministic per seed
    assert not np.array_equal(x, z)
    assert not np.array_equal(x, np.arange(1000))           # actually shuffled


def test_pagealloc_full_allocates_nothing(lib):
    a = rdp.slora_pagealloc_create(10, 3)
    try:
        out = np.empty(11, np.int32)
        with pytest.raises(rdp.SloraError) as e:
            rdp.slora_pagealloc_alloc(a, 11, out)
        assert e.value.status == 2
        assert rdp.slora_pagealloc_num_free(a) == 10
    finally:
        rdp.slora_pagealloc_destroy(a)


def test_pagealloc_free_validates_before_returning(lib):
    a = rdp.slora_pagealloc_create(10, 0)
    try:
        out = np.empty(4, np.int32)
        rdp.slora_pagealloc_alloc(a, 4, out)
        bad = np.array([out[0], out[1], 9], np.int32)           # 9 was never allocated
        with pytest.raises(rdp.SloraError):
            rdp.slora_pagealloc_free(a, 3, bad)
        assert rdp.slora_pagealloc_num_free(a) == 6             # nothing returned
        dup = np.array([out[0], out[0]], np.int32)
        with pytest.raises(rdp.SloraError):
            rdp.slora_pagealloc_free(a, 2, dup)
        assert rdp.slora_pagealloc_num_free(a) == 6
        rdp.slora_pagealloc_free(a, 4, out)                     # still all allocated
        assert rdp.slora_pagealloc_num_free(a) == 10
        with pytest.raises(rdp.SloraError):                      # double free
            rdp.slora_pagealloc_free(a, 1, out[:1].copy())
    finally:
        rdp.slora_pagealloc_destroy(a)


def test_pagealloc_kv_and_adapter_pages_interleave(lib):
    """KV blocks and adapter rows drawn from one shuffled list never collide and, taken
    together, cover the pool."""
    n = 4096
    a = rdp.slora_pagealloc_create(n, 12345)
    try:
        kv = np.empty(n // 2, np.int32)
        rdp.slora_pagealloc_alloc(a, n // 2, kv)
        ad = np.empty(n // 2, np.int32)
        rdp.slora_pagealloc_alloc(a, n // 2, ad)
        assert not set(kv.tolist()) & set(ad.tolist())
        assert sorted(kv.tolist() + ad.tolist()) == list(range(n))
        # interleaved: the adapter half is not one contiguous block
        assert np.ptp(ad) > n // 2
        rdp.slora_pagealloc_free(a, n // 2, kv)
        again = np.empty(n // 2, np.int32)
        rdp.slora_pagealloc_alloc(a, n // 2, again)
        assert set(again.tolist()) == set(kv.tolist())          # reuse of released KV slots
    finally:
        rdp.slora_pagealloc_destroy(a)


def test_pool_create_without_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    st = lib.slora_pool_create(0, 256, 16, 1, 4, 0, ctypes.byref(h))
    assert st != 0 and not h.value

"""The no-allocation entry point, slora_lora_apply_noalloc, against slora_lora_apply and
the fp64 oracle.

slora_lora_apply_noalloc is for callers that must not allocate device memory inside the
call: code whose device memory belongs to a host framework's allocator, or a serving step
that cannot absorb a cudaMalloc and the device synchronisation around it.  It keeps its
scratch (token plan, work list, partial sums) in a fixed array inside the library instead
of the pool's own scratch.  These tests call it through the C ABI:

  - on a fresh pool that never ran slora_lora_apply, with the device's free memory
    unchanged across the call;
  - twice in a row on the same inputs, each result bit for bit that of slora_lora_apply
    (the same kernels run on the same plan) and within the oracle's tolerance;
  - on exact-arithmetic inputs, bit for bit against the oracle;
  - after a larger call with other adapters, tokens and segments, so stale contents of the
    shared array cannot leak into a smaller call; also with more than 2048 adapter ids,
    where the batch runs as several plans of 2048 tokens;
  - with a batch too large for one plan in the array, which runs as smaller plans.

This file is collected last so that a run that stops at its first failure has already
run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
import rank_delta_paged_gb300 as rdp
from rank_delta_paged_gb300 import workloads as W
from rank_delta_paged_gb300.harness import PoolSession

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-3, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rdp.build.build()
    rdp.lib()


def _f16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.float16)


def _np(t):
    return t.cpu().view(torch.int16).numpy().view(np.float16)


def _inputs(w, p=0):
    x = _f16(w.x(p))
    idx = torch.from_numpy(w.token_adapter_idx).cuda()
    seg = None if w.seg_indptr is None else torch.from_numpy(w.seg_indptr).cuda()
    n_seg = 0 if seg is None else int(seg.numel() - 1)
    return x, idx, seg, n_seg


def _noalloc(s, w, p=0):
    x, idx, seg, n_seg = _inputs(w, p)
    y = _f16(w.y0(p))
    rdp.slora_lora_apply_noalloc(s.pool, p, x, y, w.T, idx, seg, n_seg)
    torch.cuda.synchronize()
    return _np(y)


def _apply(s, w, p=0):
    x, idx, seg, n_seg = _inputs(w, p)
    y = _f16(w.y0(p))
    rdp.slora_lora_apply(s.pool, p, x, y, w.T, idx, seg, n_seg)
    torch.cuda.synchronize()
    return _np(y)


def _assert_close(got, ref, what):
    ok = oracle.within_tolerance(got, ref, ATOL, RTOL)
    assert ok.all(), f"{what}: {int((~ok).sum())} elements outside tolerance"


def _bits(a):
    return a.view(np.uint16)


def test_noalloc_first_call_on_fresh_pool_allocates_nothing():
    w = W.decode_7b()
    # load the library's device code on this device first (module loading is not the call's)
    with PoolSession(w) as warm:
        warm.load(w.used_adapters())
        _noalloc(warm, w)
    with PoolSession(w) as s:
        s.load(w.used_adapters())
        x, idx, seg, n_seg = _inputs(w)
        y = _f16(w.y0())
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        rdp.slora_lora_apply_noalloc(s.pool, 0, x, y, w.T, idx, seg, n_seg)
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        assert s.device_status() == 0
        assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
        got = _np(y)
    _assert_close(got, oracle.workload_reference(w), "noalloc on a fresh pool")


@pytest.mark.parametrize("make", [
    lambda: W.decode_7b(),
    lambda: W.mixed_iteration(n_layers=1, pool_bytes=1 << 30, n_prefill=3, n_decode=200),
])
def test_noalloc_matches_apply_twice(make):
    w = make()
    p = w.n_proj - 1
    with PoolSession(w) as s:
        s.load(w.used_adapters())
        ref = _apply(s, w, p)
        outs = [_noalloc(s, w, p) for _ in range(2)]
        assert s.device_status() == 0
    want = oracle.workload_reference(w, p=p)
    for got in outs:
        assert np.array_equal(_bits(got), _bits(ref)), "differs from slora_lora_apply"
        _assert_close(got, want, "noalloc vs oracle")


def test_noalloc_exact_inputs_bit_exact():
    w = W.decode_7b(T=96, values="exact")
    with PoolSession(w) as s:
        s.load(w.used_adapters())
        got = _noalloc(s, w)
        assert s.device_status() == 0
    ref = oracle.workload_reference(w).astype(np.float16)
    assert np.array_equal(_bits(got), _bits(ref))


def test_noalloc_small_call_after_large_call():
    """A large call (many adapters, tokens, segments) leaves its plan and partials in the
    shared array; the next, smaller call (other adapters, fewer tokens, no segments) must
    not see them."""
    big = W.mixed_iteration(n_layers=1, pool_bytes=1 << 30, n_prefill=2, n_decode=300, seed=3)
    small = big.later_batch(1)
    small = W.Workload("small_after_big", big.hidden, big.n_proj, big.ranks, small.token_adapter_idx[-40:].copy(),
                       None, num_pages=big.num_pages, kv_pages=big.kv_pages, shuffle_seed=big.shuffle_seed,
                       seed=big.seed, n_layers=big.n_layers)
    with PoolSession(big) as s:
        s.load(np.union1d(big.used_adapters(), small.used_adapters()))
        _noalloc(s, big, 1)
        got = _noalloc(s, small, 2)
        ref = _apply(s, small, 2)
        assert s.device_status() == 0
    assert np.array_equal(_bits(got), _bits(ref))
    _assert_close(got, oracle.workload_reference(small, p=2), "small after large")


def test_noalloc_chunked_plans_with_many_adapter_ids():
    """More than 2048 adapter ids: the batch runs as plans of 2048 tokens each, every plan
    reusing the array."""
    n = 3000
    rng = np.random.default_rng(11)
    ranks = rng.choice(np.array([8, 16, 32, 64], np.int32), size=n)
    idx = rng.integers(-1, n, size=4500).astype(np.int32)
    w = W.Workload("noalloc_chunked", 1024, 1, ranks, idx, None, num_pages=2 * 2 * int(ranks.sum()),
                   kv_pages=0, shuffle_seed=4, seed=12)
    with PoolSession(w) as s:
        s.load(w.used_adapters())
        got = _noalloc(s, w)
        ref = _apply(s, w)
        assert s.device_status() == 0
    assert np.array_equal(_bits(got), _bits(ref))
    _assert_close(got, oracle.workload_reference(w), "chunked plans")


def test_noalloc_batch_beyond_one_plan_runs_as_smaller_plans():
    """8000 decode tokens at hidden 4096 with rank-64 adapters need about 2.2 KB of scratch
    per token, more than the 16 MiB array holds in one plan: the call runs them as smaller
    plans, bit for bit what slora_lora_apply gives and within the oracle's tolerance."""
    ranks = np.array([64, 8, 32], np.int32)
    idx = (np.arange(8000) % 3).astype(np.int32)
    w = W.Workload("noalloc_big", 4096, 1, ranks, idx, None, num_pages=2 * int(ranks.sum()) + 8,
                   kv_pages=0, shuffle_seed=1, seed=3)
    with PoolSession(w) as s:
        s.load([0, 1, 2])
        got = _noalloc(s, w)
        ref = _apply(s, w)
        assert s.device_status() == 0
    assert np.array_equal(_bits(got), _bits(ref))
    sel = np.arange(0, w.T, 7).astype(np.int32)
    _assert_close(got[sel], oracle.workload_reference(w, sel=sel), "smaller plans")

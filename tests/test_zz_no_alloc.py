"""The no-allocation entry point, slora_lora_apply_noalloc, against slora_lora_apply.

slora_lora_apply_noalloc is for callers that must not allocate device memory inside
the call: code whose device memory belongs to a host framework's allocator, or a serving
step that cannot absorb a cudaMalloc and the synchronisation around it.  It keeps its
token-plan scratch in a fixed array inside the library instead.  These tests call both
entry points through the C ABI on the same inputs, twice in a row (the second call runs
on the scratch the first one left behind), and check the outputs agree within the
tolerance the parity tests use; they also check that a batch too large for the fixed
array is refused with a clear error.  This file is collected last so that a run that
stops at its first failure has already run every other test.
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


def _both(w, p=0):
    """y from slora_lora_apply, then y from two consecutive slora_lora_apply_noalloc calls."""
    with PoolSession(w) as s:
        s.load(w.used_adapters())
        x = _f16(w.x(p))
        idx = torch.from_numpy(w.token_adapter_idx).cuda()
        seg = None if w.seg_indptr is None else torch.from_numpy(w.seg_indptr).cuda()
        n_seg = 0 if seg is None else int(seg.numel() - 1)
        y_ref = _f16(w.y0(p))
        rdp.slora_lora_apply(s.pool, p, x, y_ref, w.T, idx, seg, n_seg)
        outs = []
        for _ in range(2):
            y = _f16(w.y0(p))
            rdp.slora_lora_apply_noalloc(s.pool, p, x, y, w.T, idx, seg, n_seg)
            torch.cuda.synchronize()
            outs.append(_np(y))
        torch.cuda.synchronize()
        assert s.device_status() == 0
        return _np(y_ref), outs


@pytest.mark.parametrize("make", [
    lambda: W.decode_7b(),
    lambda: W.mixed_iteration(n_layers=1, pool_bytes=1 << 30, n_prefill=3, n_decode=200),
])
def test_noalloc_matches_apply_twice(make):
    w = make()
    ref, outs = _both(w, p=w.n_proj - 1)
    for got in outs:
        ok = oracle.within_tolerance(got, ref.astype(np.float64), ATOL, RTOL)
        assert ok.all(), f"{int((~ok).sum())} elements differ beyond tolerance"


def test_noalloc_refuses_batch_beyond_its_scratch():
    # 16384 decode tokens need about 36 * 16384 bytes of plan: more than the 512 KiB array
    ranks = np.array([16, 8], np.int32)
    idx = (np.arange(16384) % 2).astype(np.int32)
    w = W.Workload("noalloc_big", 256, 1, ranks, idx, None, num_pages=2 * int(ranks.sum()) + 8,
                   kv_pages=0, shuffle_seed=1, seed=3)
    with PoolSession(w) as s:
        s.load([0, 1])
        x, y = _f16(w.x()), _f16(w.y0())
        d_idx = torch.from_numpy(idx).cuda()
        with pytest.raises(rdp.SloraError) as e:
            rdp.slora_lora_apply_noalloc(s.pool, 0, x, y, w.T, d_idx)
        assert e.value.status == 11   # SLORA_ERR_UNSUPPORTED
        assert "static scratch" in str(e.value)
        torch.cuda.synchronize()
        assert np.array_equal(_np(y).view(np.uint16), w.y0().view(np.uint16))   # nothing launched

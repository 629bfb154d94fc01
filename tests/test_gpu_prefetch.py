"""The prefetch pipeline on the GPU: load(k+1) runs on the pool's side stream while apply(k)
runs on the caller's stream (S-LoRA: Serving Thousands of Concurrent LoRA Adapters
(explainer), "Algorithm / figure walkthrough" step 2).  Over five batches drawn from one
adapter zoo with exact-arithmetic values, every batch's output is bit for bit the oracle's,
in both load paths (zero-copy kernel and copy engines + staging ring), and each later load
starts before the earlier batch's apply ends (CUDA events on both streams)."""
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


def _f16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.float16)


@pytest.mark.parametrize("mode,staging", [(rdp.SLORA_LOAD_ZERO_COPY, 0),
                                          (rdp.SLORA_LOAD_COPY_ENGINE, 0),
                                          (rdp.SLORA_LOAD_COPY_ENGINE, 3 << 20)],
                         ids=["zero_copy", "copy_engine", "copy_engine_small_ring"])
def test_interleaved_loads_and_applies_bit_exact(mode, staging):
    base = W.decode_13b_zoo(values="exact", T=96, n_adapters=400)
    K = 5
    batches = [base] + [base.later_batch(k) for k in range(1, K)]
    need, resident = [], set()
    for b in batches:
        ids = [int(a) for a in b.used_adapters() if int(a) not in resident]
        need.append(ids)
        resident |= set(ids)
    assert all(len(n) > 0 for n in need)
    st = torch.cuda.current_stream()
    with PoolSession(base) as s:
        rdp.slora_pool_set_load_mode(s.pool, mode, staging)
        assert rdp.slora_pool_get_load_mode(s.pool)[0] == mode
        s.register(sorted(resident))
        x = _f16(base.x())
        ys = [_f16(base.y0()) for _ in range(K)]
        idx = [torch.from_numpy(b.token_adapter_idx).cuda() for b in batches]
        # a first apply (base-only tokens) sizes the pool's plan scratch, as in a serving
        # loop that is already running; that allocation synchronises the device
        none = torch.full((base.T,), -1, dtype=torch.int32, device="cuda")
        rdp.slora_lora_apply(s.pool, 0, x, _f16(base.y0()), base.T, none, None, 0, None, st)
        torch.cuda.synchronize()
        ev = lambda: torch.cuda.Event(enable_timing=True)
        begin, end, load_start = [ev() for _ in range(K)], [ev() for _ in range(K)], [ev() for _ in range(K)]
        for e in begin + end + load_start:
            e.record(st)   # creates the CUDA events (the pool records load_start again later)
        torch.cuda.synchronize()
        rdp.slora_pool_set_load_start_event(s.pool, load_start[0])
        s.load(need[0], st)
        for k in range(K):
            begin[k].record(st)
            rdp.slora_lora_apply(s.pool, 0, x, ys[k], base.T, idx[k], None, 0, None, st)
            end[k].record(st)
            if k + 1 < K:   # the next batch's adapters, on the side stream, behind apply(k)
                rdp.slora_pool_set_load_start_event(s.pool, load_start[k + 1])
                s.load(need[k + 1], st)
        torch.cuda.synchronize()
        rdp.slora_pool_set_load_start_event(s.pool, None)
        assert s.device_status() == 0
        got = [y.cpu().view(torch.int16).numpy().view(np.float16) for y in ys]
        overlapped = [load_start[k + 1].elapsed_time(end[k]) > 0 for k in range(K - 1)]
    for k, b in enumerate(batches):
        ref = oracle.workload_reference(b).astype(np.float16)
        assert np.array_equal(got[k].view(np.uint16), ref.view(np.uint16)), k
    # every later load began on the side stream before the earlier batch's apply ended
    assert all(overlapped), overlapped

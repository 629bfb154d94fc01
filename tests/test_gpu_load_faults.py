"""Failure paths of the adapter load, made on the host (no GPU fault): a load-kernel launch,
a directory-update launch, a staging copy or the staging ring's growth fails as if its CUDA
call had failed, or the page-table arena is short.  The load must take itself back (no page
lost, no adapter resident, directory cleared) and a later load of the same adapters must give
results bit for bit equal to the oracle on exact inputs (explainer, "The mechanism": adapters
move between the host store and the pool; the survey's failure-detection plan names exactly
these steps)."""
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


@pytest.fixture(autouse=True)
def _clear_injection():
    yield
    rdp.slora_debug_inject_load_fault(rdp.SLORA_FAULT_NONE, 0)


def _f16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.float16)


def _apply(s, w):
    x, y = _f16(w.x()), _f16(w.y0())
    idx = torch.from_numpy(w.token_adapter_idx).cuda()
    rdp.slora_lora_apply(s.pool, 0, x, y, w.T, idx)
    torch.cuda.synchronize()
    return y.cpu().view(torch.int16).numpy().view(np.float16)


ZC, CE = rdp.SLORA_LOAD_ZERO_COPY, rdp.SLORA_LOAD_COPY_ENGINE
CASES = [
    (ZC, rdp.SLORA_FAULT_SCATTER, 1, 6), (ZC, rdp.SLORA_FAULT_DIRECTORY, 1, 6),
    (ZC, rdp.SLORA_FAULT_ARENA, 4, 2),
    (CE, rdp.SLORA_FAULT_COPY, 1, 6), (CE, rdp.SLORA_FAULT_COPY, 7, 6),
    (CE, rdp.SLORA_FAULT_SCATTER, 3, 6), (CE, rdp.SLORA_FAULT_STAGING, 1, 6),
    (CE, rdp.SLORA_FAULT_DIRECTORY, 1, 6),
]


@pytest.mark.parametrize("mode,kind,nth,status", CASES,
                         ids=[f"{'zc' if m == ZC else 'ce'}-kind{k}-n{n}" for m, k, n, _ in CASES])
def test_failed_load_takes_itself_back(mode, kind, nth, status):
    w = W.decode_7b(values="exact", T=96, n_adapters=24)
    used = w.used_adapters()
    with PoolSession(w) as s:
        # a small staging ring: several copy + load-kernel rounds per load, and a growth
        # allocation when an adapter is larger than the ring
        rdp.slora_pool_set_load_mode(s.pool, mode, 256 << 10 if mode == CE else 0)
        s.register(used.tolist())
        free0 = rdp.slora_pool_num_free(s.pool)
        rdp.slora_debug_inject_load_fault(kind, nth)
        with pytest.raises(rdp.SloraError) as e:
            rdp.slora_adapters_load(s.pool, len(used), np.ascontiguousarray(used, np.int32), None)
        assert e.value.status == status, str(e.value)
        torch.cuda.synchronize()
        assert rdp.slora_pool_num_free(s.pool) == free0          # every page back
        assert not any(rdp.slora_adapter_is_resident(s.pool, int(a)) for a in used)
        assert s.device_status() == 0
        # the same adapters load normally afterwards, and the delta is exact
        rdp.slora_debug_inject_load_fault(rdp.SLORA_FAULT_NONE, 0)
        s.load(used)
        got = _apply(s, w)
        assert s.device_status() == 0
        assert rdp.slora_pool_num_free(s.pool) == free0 - sum(w.adapter_pages(int(a)) for a in used)
    ref = oracle.workload_reference(w).astype(np.float16)
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))


def test_injection_argument_checks():
    with pytest.raises(rdp.SloraError):
        rdp.slora_debug_inject_load_fault(99, 1)
    with pytest.raises(rdp.SloraError):
        rdp.slora_debug_inject_load_fault(rdp.SLORA_FAULT_COPY, -1)

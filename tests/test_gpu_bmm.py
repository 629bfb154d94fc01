"""GPU checks of the padded batched-GEMM comparison path (slora_lora_apply_bmm): the
same results as the oracle (bit for bit on exact-arithmetic inputs, where the custom
kernels match too) and its argument checks."""
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


def run_bmm(s, w, p=0, idx=None):
    dev = torch.device("cuda")
    idx = w.token_adapter_idx if idx is None else idx
    x = torch.from_numpy(w.x(p).view(np.int16)).to(dev).view(torch.float16)
    y = torch.from_numpy(w.y0(p).view(np.int16)).to(dev).view(torch.float16)
    idd = torch.from_numpy(np.ascontiguousarray(idx, np.int32)).to(dev)
    nb = rdp.slora_bmm_workspace_bytes(s.pool, len(idx))
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    rdp.slora_lora_apply_bmm(s.pool, p, x, y, len(idx), idd, ws, nb)
    torch.cuda.synchronize()
    return y.cpu().view(torch.int16).numpy().view(np.float16)


def test_bmm_exact_inputs_bit_exact():
    ranks = np.array([8, 16, 32, 64, 8, 16], np.int32)
    rng = np.random.default_rng(2)
    idx = rng.integers(-1, len(ranks), size=70).astype(np.int32)
    w = W.Workload("bmm_exact", 1024, 2, ranks, idx, None, num_pages=4 * 2 * int(ranks.sum()) + 32,
                   kv_pages=32, shuffle_seed=3, seed=4, values="exact")
    with PoolSession(w) as s:
        s.load(range(w.n_adapters))
        for p in range(2):
            got = run_bmm(s, w, p)
            ref = oracle.workload_reference(w, p=p).astype(np.float16)
            assert np.array_equal(got.view(np.uint16), ref.view(np.uint16)), p
        assert s.device_status() == 0


def test_bmm_normal_values_within_tolerance():
    w = W.decode_7b(T=64, seed=5)
    with PoolSession(w) as s:
        s.load(w.used_adapters())
        got = run_bmm(s, w)
        assert s.device_status() == 0
    assert oracle.within_tolerance(got, oracle.workload_reference(w), 1e-3, 1e-2).all()


def test_bmm_argument_checks():
    w = W.tiny_decode()
    with PoolSession(w) as s:
        s.load(range(w.n_adapters))
        x, y0, idx, _ = s.device_inputs(0)
        nb = rdp.slora_bmm_workspace_bytes(s.pool, w.T)
        assert nb >= w.T * 16 * 4 * w.hidden   # padded rank 16 at hidden 256
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
        with pytest.raises(rdp.SloraError) as ei:
            rdp.slora_lora_apply_bmm(s.pool, 0, x, y0, w.T, idx, ws, nb - 16)
        assert ei.value.status == 1
        with pytest.raises(rdp.SloraError):
            rdp.slora_lora_apply_bmm(s.pool, 1, x, y0, w.T, idx, ws, nb)   # one projection

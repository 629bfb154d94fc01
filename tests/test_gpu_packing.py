"""Small items sharing a unit: the last item of an adapter's tokens, with at most two tokens
and rank at most 32, shares a work group with other such items (four of rank <= 16 on
16-row slots, two of rank 17..32 on 32-row slots).  Each token's arithmetic must not depend
on its partners: its rows start on a multiple of 16, so its K steps line up as in a unit of
its own and the partners' rows add exact zeros.

  - exact-arithmetic inputs over the packing boundaries (ranks 1..33 and 64, groups of 1, 2,
    3, 9, 10, 16 and 17 tokens, partial packs, two projections): bit for bit the oracle;
  - random values: one adapter's tokens give the same bits whatever they are packed with
    (other partners, fewer partners, a batch of its own).
"""
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


def _run(s, w, p, idx, x=None, y0=None):
    x = w.x(p) if x is None else x
    y0 = w.y0(p) if y0 is None else y0
    xd, yd = _f16(x), _f16(y0)
    idd = torch.from_numpy(np.ascontiguousarray(idx, np.int32)).cuda()
    rdp.slora_lora_apply(s.pool, p, xd, yd, int(idx.shape[0]), idd)
    torch.cuda.synchronize()
    return yd.cpu().view(torch.int16).numpy().view(np.float16)


def test_packing_boundaries_bit_exact():
    ranks = np.array([1, 5, 15, 16, 17, 31, 32, 33, 64, 8, 12, 24], np.int32)
    counts = [1, 2, 3, 1, 2, 9, 10, 1, 2, 16, 17, 1]     # tokens per adapter
    idx = np.concatenate([np.full(c, a) for a, c in enumerate(counts)] + [np.full(7, -1)]).astype(np.int32)
    idx = idx[np.random.default_rng(8).permutation(idx.size)]
    w = W.Workload("packing", 1024, 2, ranks, idx, None, num_pages=2 * 4 * int(ranks.sum()) + 64,
                   kv_pages=64, shuffle_seed=3, seed=9, values="exact")
    with PoolSession(w) as s:
        s.load(range(w.n_adapters))
        for p in range(w.n_proj):
            got = _run(s, w, p, w.token_adapter_idx)
            assert s.device_status() == 0
            ref = oracle.workload_reference(w, p=p).astype(np.float16)
            assert np.array_equal(got.view(np.uint16), ref.view(np.uint16)), p


@pytest.mark.parametrize("rank", [8, 16, 24, 32])
def test_token_result_independent_of_partners(rank):
    # adapter 0 under test (two tokens), partners of the same packing class
    ranks = np.array([rank] + [8, 16, 12, 4, 24, 32, 20][:7], np.int32)
    w = W.Workload("partners", 2048, 1, ranks, np.zeros(2, np.int32), None,
                   num_pages=4 * int(ranks.sum()) + 64, kv_pages=64, shuffle_seed=2, seed=4)
    rng = np.random.default_rng(rank)
    T = 16
    # the two tokens of adapter 0 carry the same inputs in every batch; other rows differ
    xa = rng.standard_normal((2, w.hidden)).astype(np.float16)
    ya = rng.standard_normal((2, w.hidden)).astype(np.float16)
    batches = [
        np.array([0, 0] + [1, 2, 3] + [-1] * (T - 5)),            # packed with three partners
        np.array([5, 0, 6, 0] + [7] + [-1] * (T - 5)),            # other partners, other order
        np.array([0, 0] + [-1] * (T - 2)),                        # alone
        np.array([-1] * 9 + [0, 4, 0] + [-1] * (T - 12)),         # one partner, other rows
    ]
    outs = []
    with PoolSession(w) as s:
        s.load(range(w.n_adapters))
        for b in batches:
            b = b.astype(np.int32)
            x = rng.standard_normal((T, w.hidden)).astype(np.float16)
            y0 = rng.standard_normal((T, w.hidden)).astype(np.float16)
            x[b == 0], y0[b == 0] = xa, ya
            got = _run(s, w, 0, b, x, y0)
            assert s.device_status() == 0
            ref = oracle.lora_delta(x, y0, b, w.ranks, w.scaling(),
                                    [(w.factors(a)[0][0], w.factors(a)[1][0]) for a in range(w.n_adapters)])
            assert oracle.within_tolerance(got, ref).all()
            rows = np.nonzero(b == 0)[0]
            outs.append(got[rows])
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint16), outs[0].view(np.uint16))

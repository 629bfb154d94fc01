"""GPU checks of the batch planned once for several layers (slora_plan_create /
slora_plan_apply / slora_plan_destroy).

Every apply of a plan must equal slora_lora_apply_multi with the same projections, x and y
bit for bit (the same kernels over the same plan), applies of one plan must not depend on
the applies before them (the decode kernel resets its unit counter for the next launch),
and a plan must refuse to run once the pool's adapters have changed.
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


def to_np(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.float16)


def dev_f16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.float16)


def dev_i32(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


def bits(a):
    return np.ascontiguousarray(a).view(np.uint16)


def n_seg_of(w):
    return 0 if w.seg_indptr is None else len(w.seg_indptr) - 1


def via_multi(s, w, projs):
    idx, seg = dev_i32(w.token_adapter_idx), dev_i32(w.seg_indptr)
    ys = [dev_f16(w.y0(p)) for p in projs]
    rdp.slora_lora_apply_multi(s.pool, projs, [dev_f16(w.x(p)) for p in projs], ys, w.T, idx, seg, n_seg_of(w))
    torch.cuda.synchronize()
    return [to_np(y) for y in ys]


def via_plan(plan, w, projs):
    ys = [dev_f16(w.y0(p)) for p in projs]
    rdp.slora_plan_apply(plan, projs, [dev_f16(w.x(p)) for p in projs], ys)
    torch.cuda.synchronize()
    return [to_np(y) for y in ys]


def make_plan(s, w, n_slots):
    idx, seg = dev_i32(w.token_adapter_idx), dev_i32(w.seg_indptr)
    plan = rdp.slora_plan_create(s.pool, n_slots, w.T, idx, seg, n_seg_of(w))
    # the plan keeps its own copies: the caller's buffers may go away
    del idx, seg
    return plan


def assert_close(got, ref, what):
    ok = oracle.within_tolerance(got, ref, ATOL, RTOL)
    assert ok.all(), f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance"


def test_plan_decode_layers_equal_apply_multi_bit_exact():
    """Two layers of four projections over one plan of a 7B decode batch: each layer bit for
    bit the multi-projection call's, one decode launch per apply, the first layer again after
    the second unchanged, and within tolerance of the oracle."""
    base = W.decode_7b(T=256)
    w = W.Workload("decode_7b_2layers", base.hidden, 8, base.ranks, base.token_adapter_idx, None,
                   num_pages=8 * base.num_pages, kv_pages=8 * base.kv_pages, shuffle_seed=41, seed=5, n_layers=2)
    layers = [[0, 1, 2, 3], [4, 5, 6, 7]]
    with PoolSession(w) as s:
        s.load(w.used_adapters())
        ref = [via_multi(s, w, projs) for projs in layers]
        l0 = rdp.slora_pool_launch_count(s.pool)
        plan = make_plan(s, w, 4)
        assert rdp.slora_pool_launch_count(s.pool) - l0 == 1   # the plan kernel
        try:
            l1 = rdp.slora_pool_launch_count(s.pool)
            got = [via_plan(plan, w, projs) for projs in layers]
            assert rdp.slora_pool_launch_count(s.pool) - l1 == 2   # one decode launch per layer
            again = via_plan(plan, w, layers[0])
            assert s.device_status() == 0
        finally:
            rdp.slora_plan_destroy(plan)
    for li, projs in enumerate(layers):
        for j, p in enumerate(projs):
            assert np.array_equal(bits(got[li][j]), bits(ref[li][j])), (li, p)
    for j in range(4):
        assert np.array_equal(bits(again[j]), bits(got[0][j])), j
    assert_close(got[1][2], oracle.workload_reference(w, p=6), "decode layer 1, p=6")


def test_plan_mixed_layers_equal_apply_multi_bit_exact():
    """Two layers (q, k, v, o) of the mixed prefill + decode iteration over one plan, at a
    fixed segment-kernel cluster size: every projection bit for bit the multi-projection
    call's; sampled tokens within tolerance of the oracle."""
    w = W.mixed_iteration(n_layers=2, pool_bytes=2 << 30, n_prefill=4, n_decode=200)
    layers = [[0, 1, 2, 3], [4, 5, 6, 7]]
    rdp.slora_debug_set_prefill_cluster(2)
    try:
        with PoolSession(w) as s:
            s.load(w.used_adapters())
            ref = [via_multi(s, w, projs) for projs in layers]
            plan = make_plan(s, w, 4)
            try:
                got = [via_plan(plan, w, projs) for projs in layers]
                assert s.device_status() == 0
            finally:
                rdp.slora_plan_destroy(plan)
    finally:
        rdp.slora_debug_set_prefill_cluster(0)
    sel = np.unique(np.concatenate([w.decode_tokens(), np.arange(0, w.T, 37),
                                    w.seg_indptr[1:-1] - 1, w.seg_indptr[1:-1]])).astype(np.int32)
    for li, projs in enumerate(layers):
        for j, p in enumerate(projs):
            assert np.array_equal(bits(got[li][j]), bits(ref[li][j])), (li, p)
    assert_close(got[1][0][sel], oracle.workload_reference(w, p=4, sel=sel), "mixed layer 1, p=4")


def test_plan_chunked_equals_apply_bit_exact():
    """More than 2048 adapter ids: the plan holds one plan per 2048-token chunk, and every
    apply runs one decode launch per chunk, bit for bit slora_lora_apply's."""
    n = 3000
    rng = np.random.default_rng(21)
    ranks = rng.choice(np.array([8, 16, 32, 64], np.int32), size=n)
    idx = rng.integers(-1, n, size=4500).astype(np.int32)
    w = W.Workload("plan_chunked", 1024, 2, ranks, idx, None, num_pages=2 * 2 * 2 * int(ranks.sum()),
                   kv_pages=0, shuffle_seed=6, seed=13, n_layers=2)
    with PoolSession(w) as s:
        s.load(w.used_adapters())
        ref = [via_multi(s, w, [p]) for p in (0, 1)]
        plan = make_plan(s, w, 1)
        try:
            l1 = rdp.slora_pool_launch_count(s.pool)
            got = [via_plan(plan, w, [p]) for p in (0, 1)]
            assert rdp.slora_pool_launch_count(s.pool) - l1 == 2 * 3   # three chunks per apply
            assert s.device_status() == 0
        finally:
            rdp.slora_plan_destroy(plan)
    for p in (0, 1):
        assert np.array_equal(bits(got[p][0]), bits(ref[p][0])), p
    assert_close(got[1][0], oracle.workload_reference(w, p=1), "chunked plan, p=1")


def test_plan_exact_inputs_bit_exact_vs_oracle():
    """Segments of every rank and decode tokens on exact-arithmetic inputs: every
    projection of both applies equals the oracle bit for bit."""
    ranks = np.array([8, 16, 32, 64, 128, 24, 100], np.int32)
    lens = [130, 64, 257, 1, 128]
    seg_ids = [0, 2, 4, 5, 6]
    rng = np.random.default_rng(22)
    dec = rng.integers(-1, len(ranks), size=150).astype(np.int32)
    idx = np.concatenate([np.full(L, a) for a, L in zip(seg_ids, lens)] + [dec]).astype(np.int32)
    indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    w = W.Workload("plan_exact", 4096, 4, ranks, idx, indptr,
                   num_pages=2 * 2 * 4 * int(ranks.sum()), kv_pages=2 * 4 * int(ranks.sum()),
                   shuffle_seed=16, seed=17, values="exact")
    with PoolSession(w) as s:
        s.load(range(w.n_adapters))
        plan = make_plan(s, w, 2)
        try:
            got = [via_plan(plan, w, projs) for projs in ([0, 1], [3, 2])]
            assert s.device_status() == 0
        finally:
            rdp.slora_plan_destroy(plan)
    for projs, out in zip(([0, 1], [3, 2]), got):
        for j, p in enumerate(projs):
            ref = oracle.workload_reference(w, p=p)
            assert np.array_equal(bits(out[j]), bits(ref.astype(np.float16))), p


def test_plan_refuses_after_residency_change_and_wrong_slot_count():
    """A load or an eviction in the pool invalidates older plans (refused, nothing launched);
    an apply with another number of projections than the plan's is refused too."""
    w = W.tiny_decode()
    with PoolSession(w) as s:
        used = w.used_adapters().tolist()
        s.load(used)
        x, y0, idx, _ = s.device_inputs(0)
        plan = rdp.slora_plan_create(s.pool, 1, w.T, idx)
        try:
            rdp.slora_plan_apply(plan, [0], [x], [y0.clone()])
            launches0 = rdp.slora_pool_launch_count(s.pool)
            with pytest.raises(rdp.SloraError) as ei:
                rdp.slora_plan_apply(plan, [0, 0], [x, x], [y0.clone(), y0.clone()])
            assert ei.value.status == 1
            assert rdp.slora_pool_launch_count(s.pool) == launches0
            s.evict(used[:1])
            launches1 = rdp.slora_pool_launch_count(s.pool)
            with pytest.raises(rdp.SloraError) as ei:
                rdp.slora_plan_apply(plan, [0], [x], [y0.clone()])
            assert ei.value.status == 1, rdp.slora_last_error()
            assert rdp.slora_pool_launch_count(s.pool) == launches1
        finally:
            rdp.slora_plan_destroy(plan)
        rdp.slora_plan_destroy(0)   # NULL is a no-op
        # a fresh plan after the change runs
        s.load(used)
        plan = rdp.slora_plan_create(s.pool, 1, w.T, idx)
        try:
            y = y0.clone()
            rdp.slora_plan_apply(plan, [0], [x], [y])
            torch.cuda.synchronize()
            assert s.device_status() == 0
        finally:
            rdp.slora_plan_destroy(plan)
    assert_close(to_np(y), oracle.workload_reference(w), "tiny decode after reload")


def test_plan_remake_for_the_next_batch_bit_exact():
    """A plan remade for a later batch of the same shape (other token ids) applies that batch
    bit for bit as slora_lora_apply_multi does."""
    base = W.decode_7b(T=256)
    w = W.Workload("decode_7b_remake", base.hidden, 2, base.ranks, base.token_adapter_idx, None,
                   num_pages=2 * base.num_pages, kv_pages=2 * base.kv_pages, shuffle_seed=43, seed=7)
    w2 = w.later_batch(1)
    assert w2.T == w.T and not np.array_equal(w2.token_adapter_idx, w.token_adapter_idx)
    with PoolSession(w) as s:
        s.load(sorted(set(w.used_adapters().tolist()) | set(w2.used_adapters().tolist())))
        ref1 = via_multi(s, w, [0, 1])
        ref2 = via_multi(s, w2, [0, 1])
        plan = make_plan(s, w, 2)
        try:
            got1 = via_plan(plan, w, [0, 1])
            l0 = rdp.slora_pool_launch_count(s.pool)
            rdp.slora_plan_remake(plan, dev_i32(w2.token_adapter_idx))
            assert rdp.slora_pool_launch_count(s.pool) - l0 == 1   # the plan kernel only
            got2 = via_plan(plan, w2, [0, 1])
            assert s.device_status() == 0
        finally:
            rdp.slora_plan_destroy(plan)
    for j in range(2):
        assert np.array_equal(bits(got1[j]), bits(ref1[j])), j
        assert np.array_equal(bits(got2[j]), bits(ref2[j])), j


def test_plan_scaling_override_copied_and_remade():
    """A plan made with a scaling override keeps its own copy (the caller's array changes
    after the call); a remake with another override, and one with none, take effect; each
    apply bit for bit slora_lora_apply_multi with the same override, and within tolerance of
    the oracle."""
    ranks = np.array([16, 32, 8], np.int32)
    idx = np.array([0, 1, 2, 1, 0, 2, 2, 1, 0], np.int32)
    w = W.Workload("plan_scaling", 768, 2, ranks, idx, None, num_pages=2 * 2 * 2 * int(ranks.sum()),
                   kv_pages=0, shuffle_seed=2, seed=6, n_layers=2)
    first = np.array([0.5, -2.0, 3.0], np.float32)
    second = np.array([1.5, 0.25, -1.0], np.float32)
    didx = dev_i32(idx)

    def multi_with(s, p, scaling):
        y = dev_f16(w.y0(p))
        sd = None if scaling is None else torch.from_numpy(scaling).cuda()
        rdp.slora_lora_apply_multi(s.pool, [p], [dev_f16(w.x(p))], [y], w.T, didx, None, 0, sd)
        torch.cuda.synchronize()
        return to_np(y)

    with PoolSession(w) as s:
        s.load(range(w.n_adapters))
        refs = {(p, name): multi_with(s, p, sc) for p in (0, 1)
                for name, sc in (("first", first), ("second", second), ("none", None))}
        sd = torch.from_numpy(first.copy()).cuda()
        plan = rdp.slora_plan_create(s.pool, 1, w.T, didx, None, 0, sd)
        try:
            sd.fill_(7.0)   # the plan holds its own copy
            got_first = [via_plan(plan, w, [p])[0] for p in (0, 1)]
            rdp.slora_plan_remake(plan, didx, None, torch.from_numpy(second).cuda())
            got_second = [via_plan(plan, w, [p])[0] for p in (0, 1)]
            rdp.slora_plan_remake(plan, didx)
            got_none = [via_plan(plan, w, [p])[0] for p in (0, 1)]
            assert s.device_status() == 0
        finally:
            rdp.slora_plan_destroy(plan)
    for p in (0, 1):
        assert np.array_equal(bits(got_first[p]), bits(refs[(p, "first")])), p
        assert np.array_equal(bits(got_second[p]), bits(refs[(p, "second")])), p
        assert np.array_equal(bits(got_none[p]), bits(refs[(p, "none")])), p
    factors = [(w.factors(a)[0][1], w.factors(a)[1][1]) for a in range(3)]
    assert_close(got_second[1], oracle.lora_delta(w.x(1), w.y0(1), idx, ranks, second, factors), "remade override")

"""GPU checks of slora_lora_apply_multi: several projections of a layer in one call (one
token plan, one decode launch and one segment launch for all of them).

Each entry must equal the single-projection call bit for bit (decode tokens always;
segment tokens when the segment kernel runs the same cluster size, which the test hook
fixes), and match the fp64 oracle within the fp16 tolerance.
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


def singles(s, w, projs, xs):
    """One slora_lora_apply per entry: the outputs the multi call must reproduce."""
    idx, seg = dev_i32(w.token_adapter_idx), dev_i32(w.seg_indptr)
    out = []
    for p, x in zip(projs, xs):
        y = dev_f16(w.y0(p))
        s.apply(p, dev_f16(x), y, idx, seg)
        out.append(y)
    torch.cuda.synchronize()
    return [to_np(y) for y in out]


def multi(s, w, projs, xs, share_x=False):
    idx, seg = dev_i32(w.token_adapter_idx), dev_i32(w.seg_indptr)
    if share_x:
        xd = [dev_f16(xs[0])] * len(projs)
    else:
        xd = [dev_f16(x) for x in xs]
    ys = [dev_f16(w.y0(p)) for p in projs]
    n_seg = 0 if w.seg_indptr is None else len(w.seg_indptr) - 1
    rdp.slora_lora_apply_multi(s.pool, projs, xd, ys, w.T, idx, seg, n_seg)
    torch.cuda.synchronize()
    return [to_np(y) for y in ys]


def assert_close(got, ref, what):
    ok = oracle.within_tolerance(got, ref, ATOL, RTOL)
    assert ok.all(), f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance"


def test_multi_decode_equals_single_calls_bit_exact():
    """Four projections of a 7B decode batch: each output bit for bit the single call's
    (the work list is every (item, projection) pair), and within tolerance of the oracle."""
    base = W.decode_7b(T=256)
    w = W.Workload("decode_7b_4proj", base.hidden, 4, base.ranks, base.token_adapter_idx, None,
                   num_pages=4 * base.num_pages, kv_pages=4 * base.kv_pages, shuffle_seed=31, seed=3)
    projs = [0, 1, 2, 3]
    xs = [w.x(p) for p in projs]
    with PoolSession(w) as s:
        s.load(w.used_adapters())
        one = singles(s, w, projs, xs)
        launches0 = rdp.slora_pool_launch_count(s.pool)
        many = multi(s, w, projs, xs)
        assert rdp.slora_pool_launch_count(s.pool) - launches0 == 2   # one plan + one delta
        assert s.device_status() == 0
    for p in projs:
        assert np.array_equal(bits(many[p]), bits(one[p])), p
        assert_close(many[p], oracle.workload_reference(w, p=p), f"decode p={p}")


@pytest.mark.parametrize("ctas", [1, 2, 4])
def test_multi_mixed_layer_equals_single_calls_bit_exact(ctas):
    """One layer (q, k, v, o) of the mixed prefill + decode iteration in one call, at a
    fixed segment-kernel cluster size: every entry bit for bit the single call's; sampled
    tokens within tolerance of the oracle."""
    w = W.mixed_iteration(n_layers=1, pool_bytes=2 << 30)
    projs = [0, 1, 2, 3]
    xs = [w.x(p) for p in projs]
    rdp.slora_debug_set_prefill_cluster(ctas)
    try:
        with PoolSession(w) as s:
            s.load(w.used_adapters())
            one = singles(s, w, projs, xs)
            launches0 = rdp.slora_pool_launch_count(s.pool)
            many = multi(s, w, projs, xs)
            assert rdp.slora_pool_launch_count(s.pool) - launches0 == 3   # plan, delta, segments
            assert s.device_status() == 0
    finally:
        rdp.slora_debug_set_prefill_cluster(0)
    sel = np.unique(np.concatenate([w.decode_tokens(), np.arange(0, w.T, 41),
                                    w.seg_indptr[1:-1] - 1, w.seg_indptr[1:-1]])).astype(np.int32)
    for p in projs:
        assert np.array_equal(bits(many[p]), bits(one[p])), p
        assert_close(many[p][sel], oracle.workload_reference(w, p=p, sel=sel), f"mixed p={p}")


def test_multi_shared_x_and_repeated_projection():
    """q, k and v read one x buffer; a projection index may repeat with its own y."""
    w = W.mixed_iteration(n_layers=1, pool_bytes=2 << 30, n_prefill=3, n_decode=200)
    projs = [0, 1, 2, 1]
    x0 = w.x(0)
    xs = [x0] * len(projs)
    rdp.slora_debug_set_prefill_cluster(2)
    try:
        with PoolSession(w) as s:
            s.load(w.used_adapters())
            one = singles(s, w, projs, xs)
            many = multi(s, w, projs, xs, share_x=True)
            assert s.device_status() == 0
    finally:
        rdp.slora_debug_set_prefill_cluster(0)
    sel = np.unique(np.concatenate([w.decode_tokens(), np.arange(0, w.T, 29)])).astype(np.int32)
    for j, p in enumerate(projs):
        assert np.array_equal(bits(many[j]), bits(one[j])), j
        ref = oracle.workload_reference(w, p=p, sel=sel, x=x0)
        assert_close(many[j][sel], ref, f"shared x entry {j}")
    assert np.array_equal(bits(many[1]), bits(many[3]))


def test_multi_eight_entries_exact_inputs_bit_exact_vs_oracle():
    """The largest call (8 entries) on exact-arithmetic inputs with segments of every
    rank and decode tokens: every entry equals the oracle bit for bit, whatever cluster
    size the segment kernel picks."""
    ranks = np.array([8, 16, 32, 64, 128, 24, 100], np.int32)
    lens = [130, 64, 257, 1, 128]
    seg_ids = [0, 2, 4, 5, 6]
    rng = np.random.default_rng(12)
    dec = rng.integers(-1, len(ranks), size=150).astype(np.int32)
    idx = np.concatenate([np.full(L, a) for a, L in zip(seg_ids, lens)] + [dec]).astype(np.int32)
    indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    n_proj = 4
    w = W.Workload("multi_exact", 4096, n_proj, ranks, idx, indptr,
                   num_pages=2 * 2 * n_proj * int(ranks.sum()), kv_pages=2 * n_proj * int(ranks.sum()),
                   shuffle_seed=14, seed=15, values="exact")
    projs = [3, 2, 1, 0, 0, 1, 2, 3]
    xs = [w.x(p) for p in projs]
    with PoolSession(w) as s:
        s.load(range(w.n_adapters))
        many = multi(s, w, projs, xs)
        assert s.device_status() == 0
    for j, p in enumerate(projs):
        ref = oracle.workload_reference(w, p=p)
        assert np.array_equal(bits(many[j]), bits(ref.astype(np.float16))), j


@pytest.mark.parametrize("ctas", [2, 4])
def test_multi_split_units_exact_bit_exact_vs_oracle(ctas):
    """A small segment batch through a 3-entry call: 12 (tile, projection) units, so at 2
    and 4 CTAs per cluster every unit runs split in two by expand columns.  Exact inputs:
    every entry equals the oracle bit for bit, with the split and with it turned off."""
    ranks = np.array([16, 128, 40], np.int32)
    lens = [200, 190]
    rng = np.random.default_rng(21)
    dec = rng.integers(-1, len(ranks), size=20).astype(np.int32)
    idx = np.concatenate([np.full(L, a) for a, L in zip([0, 1], lens)] + [dec]).astype(np.int32)
    indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    n_proj = 3
    w = W.Workload("multi_split_exact", 4096, n_proj, ranks, idx, indptr,
                   num_pages=2 * 2 * n_proj * int(ranks.sum()), kv_pages=2 * n_proj * int(ranks.sum()),
                   shuffle_seed=22, seed=23, values="exact")
    projs = [2, 0, 1]
    xs = [w.x(p) for p in projs]
    outs = {}
    rdp.slora_debug_set_prefill_cluster(ctas)
    try:
        with PoolSession(w) as s:
            s.load(range(w.n_adapters))
            for split in (1, 0):
                rdp.slora_debug_set_prefill_split(split)
                outs[split] = multi(s, w, projs, xs)
                assert s.device_status() == 0
    finally:
        rdp.slora_debug_set_prefill_split(1)
        rdp.slora_debug_set_prefill_cluster(0)
    for j, p in enumerate(projs):
        ref = bits(oracle.workload_reference(w, p=p).astype(np.float16))
        assert np.array_equal(bits(outs[1][j]), ref), ("split", j)
        assert np.array_equal(bits(outs[0][j]), ref), ("unsplit", j)


def test_multi_argument_errors_launch_nothing():
    w = W.tiny_decode()
    with PoolSession(w) as s:
        s.load(range(w.n_adapters))
        x, y0, idx, _ = s.device_inputs(0)
        y1 = y0.clone()
        launches0 = rdp.slora_pool_launch_count(s.pool)
        bad = [
            ([], [], []),                                  # no entries
            ([0] * 9, [x] * 9, [y0.clone() for _ in range(9)]),   # more than 8
            ([0, 0], [x, x], [y0, y0]),                    # one y twice
            ([0, 0], [x, y0], [y0, y1]),                   # a y that is another entry's x
            ([0, 1], [x, x], [y0, y1]),                    # projection out of range (n_proj 1)
            ([0], [x[:, 1:]], [y0]),                       # misaligned x
        ]
        for projs, xs, ys in bad:
            with pytest.raises(rdp.SloraError) as ei:
                rdp.slora_lora_apply_multi(s.pool, projs, xs, ys, w.T, idx)
            assert ei.value.status == 1, (projs, rdp.slora_last_error())   # SLORA_ERR_INVALID_ARG
        assert rdp.slora_pool_launch_count(s.pool) == launches0
        # T = 0 is a no-op
        rdp.slora_lora_apply_multi(s.pool, [0], [x], [y0], 0, idx)
        assert rdp.slora_pool_launch_count(s.pool) == launches0

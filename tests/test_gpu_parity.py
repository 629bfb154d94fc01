"""GPU parity: libslora.so against the fp64 CPU oracle on the same seeded inputs.

Floating point: |y_gpu - ref| <= 1e-3 + 1e-2 * |ref| per element (fp16 in, fp32
accumulation, fp16 out), plus a delta-only variant (y0 = 0) where the same bound applies
to the delta itself.  Exact-arithmetic inputs and page contents: bit for bit.
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


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.float16)


def dev_f16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.float16)


def run(sess: PoolSession, p=0, idx=None, x=None, y0=None, seg="auto", scaling=None):
    w = sess.w
    x = w.x(p) if x is None else x
    y0 = w.y0(p) if y0 is None else y0
    idx = w.token_adapter_idx if idx is None else idx
    xd, yd = dev_f16(x), dev_f16(y0)
    idd = torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).cuda()
    if seg == "auto":
        seg = w.seg_indptr
    segd = None if seg is None else torch.from_numpy(np.ascontiguousarray(seg, np.int32)).cuda()
    sess.apply(p, xd, yd, idd, segd, scaling=scaling)
    torch.cuda.synchronize()
    return to_np(yd)


def assert_close(got, ref, what=""):
    ok = oracle.within_tolerance(got, ref, ATOL, RTOL)
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance; first "
                             f"{[(tuple(b), float(got[tuple(b)]), float(ref[tuple(b)])) for b in bad]}")


def session_all_loaded(w):
    s = PoolSession(w)
    s.load(range(w.n_adapters))
    return s


# ------------------------------------------------------------------ parity

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_decode_parity(seed):
    w = W.tiny_decode(seed=seed)
    with session_all_loaded(w) as s:
        got = run(s)
        assert s.device_status() == 0
    assert_close(got, oracle.workload_reference(w), "tiny_decode")


@pytest.mark.parametrize("values", ["exact"])
@pytest.mark.parametrize("make", [W.tiny_decode, lambda **k: W.decode_7b(T=96, **k),
                                  lambda **k: W.prefill_7b(n_seg=5, seg_len=136, **k)])
def test_exact_inputs_bit_exact(make, values):
    w = make(values=values)
    with session_all_loaded(w) as s:
        got = run(s)
        assert s.device_status() == 0
    ref = oracle.workload_reference(w)
    assert np.array_equal(got.view(np.uint16), ref.astype(np.float16).view(np.uint16))


def test_delta_only_variant():
    w = W.decode_7b(T=64, values="delta")
    with session_all_loaded(w) as s:
        got = run(s)
    ref = oracle.workload_reference(w)
    assert_close(got, ref, "delta-only")
    assert np.abs(ref).max() > 0.01


def test_decode_7b_full_size():
    w = W.decode_7b()
    with session_all_loaded(w) as s:
        got = run(s)
        assert s.device_status() == 0
    assert_close(got, oracle.workload_reference(w), "decode_7b")


def test_prefill_7b_full_size():
    """16 segments of 512 tokens: every output element against the oracle."""
    w = W.prefill_7b()
    with session_all_loaded(w) as s:
        got = run(s)
        assert s.device_status() == 0
    assert_close(got, oracle.workload_reference(w), "prefill_7b")


@pytest.mark.parametrize("make", [
    lambda: W.prefill_7b(values="delta"),
    lambda: W.decode_13b_zoo(values="delta"),
    lambda: W.mixed_iteration(n_layers=1, pool_bytes=2 << 30, values="delta"),
], ids=["prefill_7b", "decode_13b_zoo", "mixed_layer"])
def test_delta_only_full_configs(make):
    """y0 = 0, so the bound 1e-3 + 1e-2 |ref| applies to the delta itself (for the prefill
    path, which rounds x A to fp16, and for the decode path at 2000 pooled adapters)."""
    w = make()
    with PoolSession(w) as s:
        s.load(w.used_adapters())
        for p in range(w.n_proj):
            got = run(s, p=p)
            assert s.device_status() == 0
            ref = oracle.workload_reference(w, p=p)
            assert_close(got, ref, f"{w.name} delta-only p={p}")
            assert np.abs(ref).max() > 0.01


def test_prefill_ragged_segments():
    """Segments that are not multiples of the 128-token tile, one of a single token, and
    decode tokens before and after the segment range."""
    rng = np.random.default_rng(5)
    ranks = np.array([8, 16, 32, 64, 128, 8, 24], np.int32)
    lens = [1, 127, 129, 300, 64, 5]
    pre, post = 7, 9
    ids = [rng.integers(0, 7, pre)]
    for i, L in enumerate(lens):
        ids.append(np.full(L, i % 7))
    ids.append(rng.integers(-1, 7, post))
    idx = np.concatenate(ids).astype(np.int32)
    indptr = np.concatenate([[pre], pre + np.cumsum(lens)]).astype(np.int32)
    w = W.Workload("ragged", 1024, 1, ranks, idx, indptr, num_pages=2 * 2 * int(ranks.sum()),
                   kv_pages=2 * int(ranks.sum()), shuffle_seed=99, seed=11)
    with session_all_loaded(w) as s:
        got = run(s)
        assert s.device_status() == 0
    assert_close(got, oracle.workload_reference(w), "ragged segments")


def test_decode_13b_cold_load_then_apply():
    w = W.decode_13b_zoo()
    used = w.used_adapters()
    with PoolSession(w) as s:
        s.register(range(w.n_adapters))          # the whole zoo sits in the pinned host store
        stream = torch.cuda.current_stream()
        s.load(used, stream=stream)              # cold: fetch the batch's adapters
        got = run(s)
        assert s.device_status() == 0
        # everything else stayed on the host
        assert not rdp.slora_adapter_is_resident(s.pool, int(np.setdiff1d(np.arange(w.n_adapters), used)[0]))
    assert_close(got, oracle.workload_reference(w), "decode_13b")


def test_mixed_iteration_one_layer():
    w = W.mixed_iteration(n_layers=1, pool_bytes=2 << 30)
    used = w.used_adapters()
    with PoolSession(w) as s:
        s.load(used)
        for p in range(w.n_proj):
            got = run(s, p=p)
            assert_close(got, oracle.workload_reference(w, p=p), f"mixed p={p}")
        assert s.device_status() == 0


# ------------------------------------------------------------------ pool semantics

def test_page_gather_bit_exact_and_reload():
    w = W.decode_7b(T=32, n_adapters=12)
    with PoolSession(w) as s:
        s.load(range(w.n_adapters))
        first = {}
        for a in range(w.n_adapters):
            r = int(w.ranks[a])
            pt = np.empty(2 * r, np.int32)
            rdp.slora_adapter_pages(s.pool, a, 0, pt)
            first[a] = pt.copy()
            At, B = w.factors(a)
            want = np.concatenate([At[0], B[0]]).view(np.uint16)
            page = np.empty(w.hidden, np.uint16)
            for j in range(2 * r):
                rdp.slora_page_read(s.pool, int(pt[j]), page)
                assert np.array_equal(page, want[j]), (a, j)
        allp = np.concatenate(list(first.values()))
        assert len(np.unique(allp)) == allp.size                 # no page shared
        assert not set(allp.tolist()) & set(s.kv_pages.tolist())  # none taken from KV
        y_before = run(s)
        # evict everything, release half of the KV slots, take some free slots so the
        # reload lands elsewhere (partly on former KV slots), reload in reverse order
        s.evict(range(w.n_adapters))
        kv_half = s.kv_pages[: s.kv_pages.size // 2].copy()
        rdp.slora_pages_free(s.pool, kv_half.size, kv_half)
        hold = np.empty(97, np.int32)
        rdp.slora_pages_alloc(s.pool, 97, hold)
        s.load(range(w.n_adapters)[::-1])
        moved = 0
        for a in range(w.n_adapters):
            r = int(w.ranks[a])
            pt = np.empty(2 * r, np.int32)
            rdp.slora_adapter_pages(s.pool, a, 0, pt)
            moved += int(not np.array_equal(pt, first[a]))
            At, B = w.factors(a)
            want = np.concatenate([At[0], B[0]]).view(np.uint16)
            page = np.empty(w.hidden, np.uint16)
            for j in range(0, 2 * r, 3):
                rdp.slora_page_read(s.pool, int(pt[j]), page)
                assert np.array_equal(page, want[j])
        assert moved > 0
        y_after = run(s)
        assert np.array_equal(y_before.view(np.uint16), y_after.view(np.uint16))


def test_batch_order_invariance_bit_exact():
    w = W.decode_7b(T=200, n_adapters=20)
    perm = np.random.default_rng(3).permutation(w.T)
    with session_all_loaded(w) as s:
        y = run(s)
        yp = run(s, idx=w.token_adapter_idx[perm], x=w.x()[perm], y0=w.y0()[perm])
    assert np.array_equal(yp.view(np.uint16), y[perm].view(np.uint16))


def test_zero_B_leaves_y_unchanged():
    w = W.tiny_decode(seed=4)
    w.prefetch_factors(range(w.n_adapters))
    for a in range(w.n_adapters):
        At, B = w.factors(a)
        B[...] = 0
    with session_all_loaded(w) as s:
        got = run(s)
    assert np.array_equal(got.view(np.uint16), w.y0().view(np.uint16))


def test_base_only_tokens_and_errors_are_skipped():
    w = W.tiny_decode(seed=8, T=16)
    with PoolSession(w) as s:
        s.load([0, 1, 2])                       # adapter 3 stays on the host
        idx = w.token_adapter_idx.copy()
        idx[0] = -1
        idx[1] = 3                               # not resident
        got = run(s, idx=idx)
        assert s.device_status() == rdp_dev("NOT_RESIDENT")
        y0 = w.y0()
        assert np.array_equal(got[0].view(np.uint16), y0[0].view(np.uint16))
        assert np.array_equal(got[1].view(np.uint16), y0[1].view(np.uint16))
        keep = idx != 3
        ref = oracle.workload_reference(w, sel=np.nonzero(keep)[0].astype(np.int32))
        # reference for the kept tokens with the modified map
        ref = oracle.lora_delta(w.x(), y0, np.where(keep, idx, -1).astype(np.int32), w.ranks,
                                w.scaling(), [(w.factors(a)[0][0], w.factors(a)[1][0]) for a in range(4)])
        assert_close(got, ref, "base-only/skip")
        idx[2] = 17                              # beyond max_adapters
        run(s, idx=idx)
        assert s.device_status() in (rdp_dev("BAD_ADAPTER"), rdp_dev("NOT_RESIDENT"))
        assert s.device_status() == 0           # cleared by the read


def rdp_dev(name):
    return {"BAD_ADAPTER": 1, "NOT_RESIDENT": 2, "BAD_PAGE": 3, "BAD_SEGMENT": 4}[name]


def test_odd_ranks_and_ragged_token_counts():
    ranks = np.array([1, 3, 8, 17, 128, 40], np.int32)
    for T in (1, 2, 33, 257):
        idx = np.random.default_rng(T).integers(-1, len(ranks), T).astype(np.int32)
        w = W.Workload(f"odd{T}", 512, 1, ranks, idx, None, num_pages=4 * int(ranks.sum()),
                       kv_pages=int(ranks.sum()), shuffle_seed=5, seed=T)
        with session_all_loaded(w) as s:
            got = run(s)
            assert s.device_status() == 0
        assert_close(got, oracle.workload_reference(w), f"odd ranks T={T}")


def test_scaling_override_and_projection_select():
    ranks = np.array([16, 32, 8], np.int32)
    idx = np.array([0, 1, 2, 1, 0, 2, 2], np.int32)
    w = W.Workload("proj3", 768, 3, ranks, idx, None, num_pages=2 * 3 * 2 * int(ranks.sum()),
                   kv_pages=0, shuffle_seed=1, seed=4)
    override = np.array([0.5, -2.0, 3.0], np.float32)
    with session_all_loaded(w) as s:
        for p in range(3):
            got = run(s, p=p)
            assert_close(got, oracle.workload_reference(w, p=p), f"proj {p}")
        sd = torch.from_numpy(override).cuda()
        got = run(s, p=2, scaling=sd)
    factors = [(w.factors(a)[0][2], w.factors(a)[1][2]) for a in range(3)]
    ref = oracle.lora_delta(w.x(2), w.y0(2), idx, ranks, override, factors)
    assert_close(got, ref, "scaling override")


def test_empty_batch_is_noop():
    w = W.tiny_decode()
    with session_all_loaded(w) as s:
        y = torch.zeros(1, w.hidden, dtype=torch.float16, device="cuda")
        x = torch.zeros_like(y)
        idx = torch.zeros(1, dtype=torch.int32, device="cuda")
        rdp.slora_lora_apply(s.pool, 0, x, y, 0, idx)
        torch.cuda.synchronize()
        assert int(y.abs().sum()) == 0


def test_pool_full_loads_nothing():
    w = W.decode_7b(T=8, n_adapters=10)
    with PoolSession(w) as s:
        free = rdp.slora_pool_num_free(s.pool)
        hold = np.empty(free - 10, np.int32)
        rdp.slora_pages_alloc(s.pool, free - 10, hold)
        with pytest.raises(rdp.SloraError) as e:
            s.load(range(w.n_adapters))
        assert e.value.status == 2
        assert rdp.slora_pool_num_free(s.pool) == 10
        assert not any(rdp.slora_adapter_is_resident(s.pool, a) for a in range(w.n_adapters))


def test_segment_edge_cases():
    """A segment whose adapter has rank > 128 (routed to the decode path), a base-only
    segment (-1), an empty segment, and single-token segments."""
    ranks = np.array([8, 200, 16, 256], np.int32)
    lens = [130, 0, 70, 1, 1, 40]
    seg_adapter = [1, 2, -1, 0, 3, 1]
    idx = np.concatenate([np.full(L, a) for L, a in zip(lens, seg_adapter)] +
                         [np.array([0, 1, 2, 3, -1], np.int32)]).astype(np.int32)
    indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    w = W.Workload("seg_edges", 512, 1, ranks, idx, indptr, num_pages=2 * 2 * int(ranks.sum()),
                   kv_pages=int(ranks.sum()), shuffle_seed=3, seed=21)
    with session_all_loaded(w) as s:
        got = run(s)
        assert s.device_status() == 0
    assert_close(got, oracle.workload_reference(w), "segment edges")


def test_segment_with_mixed_adapters_is_rejected():
    ranks = np.array([16, 32], np.int32)
    idx = np.array([0] * 100 + [1] + [0] * 27 + [1] * 50, np.int32)   # first 128-token tile mixed
    indptr = np.array([0, 128, 178], np.int32)
    w = W.Workload("seg_mixed", 256, 1, ranks, idx, indptr, num_pages=8 * int(ranks.sum()),
                   kv_pages=0, shuffle_seed=0, seed=2)
    with session_all_loaded(w) as s:
        got = run(s)
        assert s.device_status() == rdp_dev("BAD_SEGMENT")
    y0 = w.y0()
    # the mixed segment is skipped (y unchanged); the second segment is computed
    assert np.array_equal(got[:128].view(np.uint16), y0[:128].view(np.uint16))
    assert_close(got[128:], oracle.workload_reference(w, sel=np.arange(128, 178, dtype=np.int32)),
                 "second segment")


def test_segment_mixed_in_a_later_tile_is_rejected_whole():
    """A segment of 300 tokens whose token 250 names another adapter: every token of the
    segment keeps y0, whichever tiles the kernel cuts the segment into; the next segment is
    computed."""
    ranks = np.array([16, 32], np.int32)
    idx = np.array([0] * 250 + [1] + [0] * 49 + [1] * 50, np.int32)
    indptr = np.array([0, 300, 350], np.int32)
    w = W.Workload("seg_mixed_late", 256, 1, ranks, idx, indptr, num_pages=8 * int(ranks.sum()),
                   kv_pages=0, shuffle_seed=0, seed=4)
    with session_all_loaded(w) as s:
        got = run(s)
        assert s.device_status() == rdp_dev("BAD_SEGMENT")
    y0 = w.y0()
    assert np.array_equal(got[:300].view(np.uint16), y0[:300].view(np.uint16))
    assert_close(got[300:], oracle.workload_reference(w, sel=np.arange(300, 350, dtype=np.int32)),
                 "second segment")


def test_prefill_exact_all_ranks_bit_exact():
    """Exact-arithmetic inputs through the tensor-core path for every rank class and a
    hidden size that is not a multiple of the 256-column tile."""
    ranks = np.array([8, 16, 24, 32, 64, 100, 128], np.int32)
    lens = [128, 129, 64, 200, 17, 128, 256]
    idx = np.concatenate([np.full(L, i) for i, L in enumerate(lens)]).astype(np.int32)
    indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    w = W.Workload("prefill_exact", 704, 1, ranks, idx, indptr, num_pages=2 * 2 * int(ranks.sum()),
                   kv_pages=int(ranks.sum()), shuffle_seed=8, seed=5, values="exact")
    with session_all_loaded(w) as s:
        got = run(s)
        assert s.device_status() == 0
    ref = oracle.workload_reference(w)
    assert np.array_equal(got.view(np.uint16), ref.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("ctas", [1, 2, 4, 8])
def test_prefill_every_cluster_size_bit_exact(ctas):
    """The segment kernel with 1, 2, 4 and 8 CTAs per cluster on exact-arithmetic inputs
    (every partial sum an integer, so the cross-CTA sum of the shrink partials is exact in
    any order): hidden slices, the partial-product exchange, full tiles stored by tensor
    map and ragged last tiles stored row by row, next to decode tokens."""
    ranks = np.array([8, 16, 24, 32, 64, 100, 128], np.int32)
    lens = [128, 129, 64, 200, 17, 256, 300]
    idx = np.concatenate([np.full(L, i) for i, L in enumerate(lens)] +
                         [np.array([3, -1, 6, 0], np.int32)]).astype(np.int32)
    indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    w = W.Workload("prefill_clusters", 4096, 1, ranks, idx, indptr, num_pages=2 * 2 * int(ranks.sum()),
                   kv_pages=int(ranks.sum()), shuffle_seed=4, seed=6, values="exact")
    rdp.slora_debug_set_prefill_cluster(ctas)
    try:
        with session_all_loaded(w) as s:
            got = run(s)
            assert s.device_status() == 0
    finally:
        rdp.slora_debug_set_prefill_cluster(0)
    ref = oracle.workload_reference(w)
    assert np.array_equal(got.view(np.uint16), ref.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("ctas", [2, 8])
def test_prefill_cluster_normal_values(ctas):
    """Normal-valued inputs at a forced cluster size: within the fp16 tolerance."""
    w = W.prefill_7b(n_seg=5, seg_len=200)
    rdp.slora_debug_set_prefill_cluster(ctas)
    try:
        with session_all_loaded(w) as s:
            got = run(s)
            assert s.device_status() == 0
    finally:
        rdp.slora_debug_set_prefill_cluster(0)
    assert_close(got, oracle.workload_reference(w), f"prefill, {ctas} CTAs per cluster")


@pytest.mark.parametrize("hidden,ctas", [(1024, 8), (768, 4)])
def test_prefill_split_with_few_column_tiles_exact(hidden, ctas):
    """CTAs with only 2 (hidden 1024 at 8 CTAs per cluster) or 3 (hidden 768 at 4) column
    tiles of 64: units split in at most 2 parts, unevenly at 3 tiles.  Exact-arithmetic
    inputs, a handful of units: y equals the oracle bit for bit, split or not."""
    ranks = np.array([8, 64, 128], np.int32)
    lens = [128, 100, 256]
    idx = np.concatenate([np.full(L, i) for i, L in enumerate(lens)]).astype(np.int32)
    indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    w = W.Workload("prefill_few_tiles", hidden, 1, ranks, idx, indptr, num_pages=2 * 2 * int(ranks.sum()),
                   kv_pages=int(ranks.sum()), shuffle_seed=31, seed=32, values="exact")
    ref = oracle.workload_reference(w).astype(np.float16).view(np.uint16)
    rdp.slora_debug_set_prefill_cluster(ctas)
    try:
        with session_all_loaded(w) as s:
            for split in (1, 0):
                rdp.slora_debug_set_prefill_split(split)
                got = run(s)
                assert s.device_status() == 0
                assert np.array_equal(got.view(np.uint16), ref), split
    finally:
        rdp.slora_debug_set_prefill_split(1)
        rdp.slora_debug_set_prefill_cluster(0)


@pytest.mark.parametrize("ctas", [4, 8])
def test_prefill_last_round_split_matches_unsplit_bit_for_bit(ctas):
    """More units than clusters (44 against 38 clusters of 4 CTAs, or about 19 of 8): the
    units of the last, partial round are split by expand columns over the clusters that
    round would leave idle.  Normal-valued inputs: y bit for bit the unsplit kernel's at
    the same cluster size, and within the tolerance of the oracle."""
    w = W.prefill_7b(n_seg=11, seg_len=512)   # 44 units, ranks 8..128
    outs = []
    rdp.slora_debug_set_prefill_cluster(ctas)
    try:
        with session_all_loaded(w) as s:
            for split in (1, 0):
                rdp.slora_debug_set_prefill_split(split)
                outs.append(run(s))
                assert s.device_status() == 0
    finally:
        rdp.slora_debug_set_prefill_split(1)
        rdp.slora_debug_set_prefill_cluster(0)
    assert np.array_equal(outs[0].view(np.uint16), outs[1].view(np.uint16))
    assert_close(outs[0], oracle.workload_reference(w), f"last-round split, {ctas} CTAs per cluster")


@pytest.mark.parametrize("ctas", [0, 1, 2, 4])
def test_prefill_split_units_match_unsplit_bit_for_bit(ctas):
    """A batch of fewer 128-token units than resident clusters runs every unit split by
    expand columns (in 4 parts against 76 or 152 clusters, in 2 against 38; each part
    repeats the shrink on its own cluster): normal-valued inputs give y bit for bit equal
    to the unsplit kernel's at the same cluster size, and within the tolerance of the
    oracle."""
    w = W.prefill_7b(n_seg=6, seg_len=300)   # 18 units, ragged last tiles, ranks 8..128
    outs = []
    rdp.slora_debug_set_prefill_cluster(ctas)
    try:
        with session_all_loaded(w) as s:
            for split in (1, 0):
                rdp.slora_debug_set_prefill_split(split)
                outs.append(run(s))
                assert s.device_status() == 0
    finally:
        rdp.slora_debug_set_prefill_split(1)
        rdp.slora_debug_set_prefill_cluster(0)
    assert np.array_equal(outs[0].view(np.uint16), outs[1].view(np.uint16))
    assert_close(outs[0], oracle.workload_reference(w), f"split prefill, {ctas} CTAs per cluster")


def test_load_of_more_adapters_than_one_launch_carries():
    """600 adapters in one load call: two launches of the load kernel (at most 512 adapters
    each), which read the pinned store directly; pages bit-exact on both sides of the
    split, and a batch over all of them matches the oracle."""
    n = 600
    ranks = np.full(n, 8, np.int32)
    rng = np.random.default_rng(5)
    idx = rng.integers(0, n, size=256).astype(np.int32)
    w = W.Workload("many_adapters", 256, 1, ranks, idx, None, num_pages=2 * 2 * 8 * n, kv_pages=2 * 8 * n,
                   shuffle_seed=9, seed=4)
    with session_all_loaded(w) as s:
        for a in (0, 1, 511, 512, 513, 599):
            pt = np.empty(16, np.int32)
            rdp.slora_adapter_pages(s.pool, a, 0, pt)
            At, B = w.factors(a)
            want = np.concatenate([At[0], B[0]]).view(np.uint16)
            page = np.empty(w.hidden, np.uint16)
            for j in range(16):
                rdp.slora_page_read(s.pool, int(pt[j]), page)
                assert np.array_equal(page, want[j]), (a, j)
        got = run(s)
        assert s.device_status() == 0
    assert_close(got, oracle.workload_reference(w), "600 adapters")


def test_decode_large_ranks_and_long_groups_bit_exact():
    """Decode ranks 1 to 1024 (every rank bucket, items of several rank units), an adapter
    holding 40 tokens (three items), base-only tokens; exact-arithmetic inputs, so the
    kernel equals the oracle bit for bit."""
    ranks = np.array([1, 2, 3, 5, 8, 13, 16, 31, 64, 100, 128, 129, 200, 256, 512, 1024], np.int32)
    rng = np.random.default_rng(3)
    idx = rng.integers(-1, len(ranks), size=200).astype(np.int32)
    idx[rng.choice(200, 40, replace=False)] = 6
    w = W.Workload("decode_ranks", 1024, 1, ranks, idx, None, num_pages=4 * int(ranks.sum()) + 64,
                   kv_pages=64, shuffle_seed=5, seed=6, values="exact")
    with session_all_loaded(w) as s:
        got = run(s)
        assert s.device_status() == 0
    ref = oracle.workload_reference(w).astype(np.float16)
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))


def test_prefill_many_segments_bit_exact():
    """40 segments (more than the 32 the segment scheduler sorts by rank, so units are
    dealt in order), ragged lengths and mixed ranks, beside decode tokens; exact inputs,
    so the result equals the oracle bit for bit."""
    ranks = np.array([8, 16, 24, 32, 64, 100, 128, 8], np.int32)
    rng = np.random.default_rng(40)
    lens = rng.integers(1, 300, size=40)
    seg_ad = rng.integers(0, len(ranks), size=40)
    dec = rng.integers(-1, len(ranks), size=64)
    idx = np.concatenate([np.full(L, a) for a, L in zip(seg_ad, lens)] + [dec]).astype(np.int32)
    indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    w = W.Workload("many_segments", 1024, 1, ranks, idx, indptr, num_pages=4 * int(ranks.sum()) + 64,
                   kv_pages=64, shuffle_seed=6, seed=7, values="exact")
    with session_all_loaded(w) as s:
        got = run(s)
        assert s.device_status() == 0
    ref = oracle.workload_reference(w).astype(np.float16)
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))

"""Seeded synthetic inputs for the paged heterogeneous-rank LoRA delta.

This module draws numbers and nothing else: adapter ranks, fp16 LoRA factors,
token -> adapter maps, prefill segment boundaries, activations ``x`` and base
outputs ``y0``.  It holds none of the delta's arithmetic, so both the CUDA path
and the CPU oracle consume the arrays it returns without sharing any compute
code.  It imports neither the compiled library nor the oracle.

Shapes follow the S-LoRA pages: ``A`` is ``d_in x r`` and ``B`` is ``r x d_out``
(S-LoRA: Serving Thousands of Concurrent LoRA Adapters (explainer), "What this
paper explains"); ``A`` is handed out transposed, ``At[p][j]`` = column ``j`` of
``A`` for projection ``p``, because one pool page holds one hidden-length row.

Every stream of random numbers has its own child seed (``numpy.random.default_rng``
seeded with ``[seed, stream, index]``) so that one adapter's factors, or one
projection's activations, can be drawn without drawing the others:

  stream 0 : ranks, token ids, prefill lengths (one generator, in that order)
  stream 1 : adapter ``a`` factors At then B, all projections   ([seed, 1, a])
  stream 2 : projection ``p`` activations x                     ([seed, 2, p])
  stream 3 : projection ``p`` base outputs y0                   ([seed, 3, p])
"""
from __future__ import annotations

import dataclasses
import math
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

RANKS_DECODE = (8, 16, 32, 64)
RANKS_WIDE = (8, 16, 32, 64, 128)


def zipf_ids(rng: np.random.Generator, n_ids: int, size: int, alpha: float) -> np.ndarray:
    """Ids in [0, n_ids) with P(id = k-1) proportional to k**-alpha, k = 1..n_ids."""
    k = np.arange(1, n_ids + 1, dtype=np.float64)
    p = k ** (-alpha)
    p /= p.sum()
    return rng.choice(n_ids, size=size, p=p).astype(np.int32)


@dataclasses.dataclass
class Workload:
    """One seeded batch: adapter zoo, token map, segments and pool geometry.

    values:
      "normal" -- x ~ N(0,1), At ~ U(+-1/sqrt(d)), B ~ N(0, 0.02), y0 ~ N(0,1)
      "exact"  -- small integers for x and y0, {-1, 0, +1} factors with at most
                  four nonzeros per row: every partial sum is an integer below
                  2**24 and ``x.At`` fits fp16 exactly, so fp32 accumulation is
                  exact and any correct implementation rounds the same value.
      "delta"  -- as "normal" but y0 = 0, so the tolerance bounds the delta alone.
    """

    name: str
    hidden: int
    n_proj: int
    ranks: np.ndarray               # int32 [n_adapters]
    token_adapter_idx: np.ndarray   # int32 [T]; -1 = base only
    seg_indptr: Optional[np.ndarray]  # int32 [n_seg + 1] or None
    num_pages: int                  # pool slots (adapter + KV)
    kv_pages: int                   # slots taken by the KV side before any adapter loads
    shuffle_seed: int               # pool free-list permutation seed (0 = in order)
    seed: int = 0
    values: str = "normal"
    n_layers: int = 1               # projections per layer = n_proj // n_layers
    alpha: float = 1.0              # Zipf exponent of the token map's adapter ids

    _factor_cache: Dict[int, Tuple[np.ndarray, np.ndarray]] = dataclasses.field(
        default_factory=dict, repr=False)

    # ---- derived sizes -------------------------------------------------
    @property
    def n_adapters(self) -> int:
        return int(self.ranks.shape[0])

    @property
    def T(self) -> int:
        return int(self.token_adapter_idx.shape[0])

    @property
    def n_seg(self) -> int:
        return 0 if self.seg_indptr is None else int(self.seg_indptr.shape[0] - 1)

    def scaling(self) -> np.ndarray:
        """Per-adapter scaling 16 / r as float32 (a power of two for every rank used)."""
        return (16.0 / self.ranks.astype(np.float64)).astype(np.float32)

    def used_adapters(self) -> np.ndarray:
        ids = self.token_adapter_idx
        return np.unique(ids[ids >= 0]).astype(np.int32)

    def adapter_pages(self, a: int) -> int:
        return 2 * int(self.ranks[a]) * self.n_proj

    def later_batch(self, k: int) -> "Workload":
        """The k-th later batch served from the same adapter zoo and pool: the same ranks,
        factors, pool geometry, segment lengths and token count, the same x and y0, and new
        Zipf(alpha) adapter ids (seeded by the workload's seed and k): one id per prefill
        segment (all its tokens) and one per decode token."""
        rng = np.random.default_rng([self.seed, 100 + int(k)])
        if self.seg_indptr is None or self.n_seg == 0:
            ids = zipf_ids(rng, self.n_adapters, self.T, self.alpha)
        else:
            lo, hi = int(self.seg_indptr[0]), int(self.seg_indptr[-1])
            req = zipf_ids(rng, self.n_adapters, self.n_seg + self.T - (hi - lo), self.alpha)
            lens = np.diff(self.seg_indptr)
            ids = np.concatenate([req[self.n_seg:self.n_seg + lo], np.repeat(req[:self.n_seg], lens),
                                  req[self.n_seg + lo:]]).astype(np.int32)
        return Workload(f"{self.name}_next{k}", self.hidden, self.n_proj, self.ranks, ids, self.seg_indptr,
                        num_pages=self.num_pages, kv_pages=self.kv_pages,
                        shuffle_seed=self.shuffle_seed, seed=self.seed, values=self.values,
                        n_layers=self.n_layers, alpha=self.alpha)

    # ---- factors -------------------------------------------------------
    def factors(self, a: int, cache: bool = True) -> Tuple[np.ndarray, np.ndarray]:
        """(At, B) for adapter ``a``, each fp16 [n_proj][r][hidden], C-contiguous."""
        if a in self._factor_cache:
            return self._factor_cache[a]
        r = int(self.ranks[a])
        d = self.hidden
        rng = np.random.default_rng([self.seed, 1, int(a)])
        shape = (self.n_proj, r, d)
        if self.values == "exact":
            At = _sparse_pm1(rng, shape)
            B = _sparse_pm1(rng, shape)
        else:
            bound = 1.0 / math.sqrt(d)
            At = rng.random(shape, dtype=np.float32)
            At *= 2.0 * bound
            At -= bound
            At = At.astype(np.float16)
            B = rng.standard_normal(shape, dtype=np.float32)
            B *= 0.02
            B = B.astype(np.float16)
        if cache:
            self._factor_cache[a] = (At, B)
        return At, B

    def prefetch_factors(self, ids: Sequence[int], threads: int = 0) -> None:
        """Draw (and cache) the factors of ``ids`` on a thread pool."""
        todo = [int(a) for a in ids if int(a) not in self._factor_cache]
        if not todo:
            return
        threads = threads or min(16, len(todo))
        with ThreadPoolExecutor(max_workers=threads) as ex:
            for a, fac in zip(todo, ex.map(lambda a: self.factors(a, cache=False), todo)):
                self._factor_cache[a] = fac

    # ---- activations ---------------------------------------------------
    def x(self, p: int = 0) -> np.ndarray:
        rng = np.random.default_rng([self.seed, 2, int(p)])
        if self.values == "exact":
            return rng.integers(-3, 4, size=(self.T, self.hidden)).astype(np.float16)
        v = rng.standard_normal((self.T, self.hidden), dtype=np.float32)
        return v.astype(np.float16)

    def y0(self, p: int = 0) -> np.ndarray:
        if self.values == "delta":
            return np.zeros((self.T, self.hidden), dtype=np.float16)
        rng = np.random.default_rng([self.seed, 3, int(p)])
        if self.values == "exact":
            return rng.integers(-64, 65, size=(self.T, self.hidden)).astype(np.float16)
        v = rng.standard_normal((self.T, self.hidden), dtype=np.float32)
        return v.astype(np.float16)

    def decode_tokens(self) -> np.ndarray:
        """Token indices outside the prefill segment range."""
        t = np.arange(self.T, dtype=np.int32)
        if self.seg_indptr is None or self.n_seg == 0:
            return t
        lo, hi = int(self.seg_indptr[0]), int(self.seg_indptr[-1])
        return t[(t < lo) | (t >= hi)]


def _sparse_pm1(rng: np.random.Generator, shape: Tuple[int, int, int]) -> np.ndarray:
    """Rows with at most four nonzero entries, each -1 or +1 (columns drawn with
    replacement, so a repeated column keeps the last sign drawn)."""
    P, r, d = shape
    out = np.zeros(shape, dtype=np.float16)
    nnz = min(4, d)
    cols = rng.integers(0, d, size=(P, r, nnz))
    signs = np.where(rng.random((P, r, nnz)) < 0.5, -1.0, 1.0).astype(np.float16)
    np.put_along_axis(out, cols, signs, axis=2)
    return out


# ---------------------------------------------------------------------------
# The five workloads.  Names say what they are; sizes are in the constructors.
# ---------------------------------------------------------------------------

def tiny_decode(seed: int = 0, values: str = "normal", T: int = 8) -> Workload:
    """hidden 256, 4 adapters of ranks {8, 8, 16, 16}, 256-page shuffled pool, 8 tokens."""
    rng = np.random.default_rng([seed, 0])
    ranks = np.array([8, 8, 16, 16], dtype=np.int32)
    ids = rng.integers(0, 4, size=T).astype(np.int32)
    return Workload("tiny_decode_h256_a4_t8", 256, 1, ranks, ids, None,
                    num_pages=256, kv_pages=64, shuffle_seed=seed * 7919 + 11,
                    seed=seed, values=values)


def decode_7b(seed: int = 0, values: str = "normal", T: int = 256, n_adapters: int = 100,
              hidden: int = 4096, alpha: float = 1.0, n_layers: int = 1) -> Workload:
    """hidden 4096, 100 adapters of ranks U{8,16,32,64}, 256 decode tokens, Zipf(1) ids;
    n_layers layers of one projection each (the same batch through every layer).

    Pool: twice the zoo's pages, the other half held by KV, randomly interleaved.
    """
    rng = np.random.default_rng([seed, 0])
    ranks = rng.choice(np.array(RANKS_DECODE, dtype=np.int32), size=n_adapters)
    ids = zipf_ids(rng, n_adapters, T, alpha)
    zoo_pages = int(2 * ranks.sum()) * n_layers
    suffix = f"_l{n_layers}" if n_layers > 1 else ""
    return Workload(f"decode_7b_h{hidden}_a{n_adapters}_t{T}_zipf{alpha:g}{suffix}", hidden, n_layers, ranks,
                    ids, None, num_pages=2 * zoo_pages, kv_pages=zoo_pages,
                    shuffle_seed=seed * 7919 + 13, seed=seed, values=values, alpha=alpha, n_layers=n_layers)


def prefill_7b(seed: int = 0, values: str = "normal", n_seg: int = 16, seg_len: int = 512,
               hidden: int = 4096, ranks: Optional[Sequence[int]] = None, n_layers: int = 1) -> Workload:
    """hidden 4096, 16 segments x 512 tokens, segment i on adapter i, ranks cycled over
    {8, 16, 32, 64, 128}; n_layers layers of one projection each.  Pool interleaved with KV
    as in decode_7b."""
    if ranks is None:
        ranks = [RANKS_WIDE[i % len(RANKS_WIDE)] for i in range(n_seg)]
    ranks = np.asarray(ranks, dtype=np.int32)
    assert ranks.shape[0] == n_seg
    ids = np.repeat(np.arange(n_seg, dtype=np.int32), seg_len)
    indptr = (np.arange(n_seg + 1, dtype=np.int32) * seg_len).astype(np.int32)
    zoo_pages = int(2 * ranks.sum()) * n_layers
    suffix = f"_l{n_layers}" if n_layers > 1 else ""
    return Workload(f"prefill_7b_h{hidden}_s{n_seg}x{seg_len}{suffix}", hidden, n_layers, ranks, ids, indptr,
                    num_pages=2 * zoo_pages, kv_pages=zoo_pages,
                    shuffle_seed=seed * 7919 + 17, seed=seed, values=values, n_layers=n_layers)


def decode_13b_zoo(seed: int = 0, values: str = "normal", T: int = 512, n_adapters: int = 2000,
                   hidden: int = 5120, alpha: float = 0.5, n_layers: int = 1) -> Workload:
    """hidden 5120, 2000 adapters of ranks U{8,16,32,64} in the host store, 512 decode
    tokens with Zipf(0.5) ids; the pool starts cold and the batch's adapters are loaded;
    n_layers layers of one projection each (the same batch through every layer)."""
    rng = np.random.default_rng([seed, 0])
    ranks = rng.choice(np.array(RANKS_DECODE, dtype=np.int32), size=n_adapters)
    ids = zipf_ids(rng, n_adapters, T, alpha)
    zoo_pages = int(2 * ranks.sum()) * n_layers
    suffix = f"_l{n_layers}" if n_layers > 1 else ""
    return Workload(f"decode_13b_h{hidden}_a{n_adapters}_t{T}_zipf{alpha:g}{suffix}", hidden, n_layers, ranks,
                    ids, None, num_pages=2 * zoo_pages, kv_pages=zoo_pages,
                    shuffle_seed=seed * 7919 + 19, seed=seed, values=values, alpha=alpha, n_layers=n_layers)


def mixed_iteration(seed: int = 0, values: str = "normal", n_layers: int = 32,
                    n_adapters: int = 1000, hidden: int = 4096, n_prefill: int = 8,
                    prefill_len: Tuple[int, int] = (256, 1024), n_decode: int = 384,
                    pool_bytes: int = 40 << 30, alpha: float = 1.0) -> Workload:
    """32 layers x {q,k,v,o} at hidden 4096 (128 projections), 1000 adapters of ranks
    U{8,...,128}; 8 prefill requests of U[256, 1024] tokens plus 384 decode tokens, one
    Zipf(1) adapter id per request; a 40 GiB pool of hidden-length fp16 pages with half of
    the slots held by KV in random interleaving."""
    rng = np.random.default_rng([seed, 0])
    ranks = rng.choice(np.array(RANKS_WIDE, dtype=np.int32), size=n_adapters)
    req_ids = zipf_ids(rng, n_adapters, n_prefill + n_decode, alpha)
    lens = rng.integers(prefill_len[0], prefill_len[1] + 1, size=n_prefill).astype(np.int32)
    ids = np.concatenate([np.repeat(req_ids[:n_prefill], lens), req_ids[n_prefill:]]).astype(np.int32)
    indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    num_pages = pool_bytes // (hidden * 2)
    return Workload(f"mixed_iteration_h{hidden}_l{n_layers}x4_a{n_adapters}", hidden,
                    4 * n_layers, ranks, ids, indptr, num_pages=int(num_pages),
                    kv_pages=int(num_pages // 2), shuffle_seed=seed * 7919 + 23, seed=seed,
                    values=values, n_layers=n_layers, alpha=alpha)


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "decode_7b": decode_7b,
    "prefill_7b": prefill_7b,
    "decode_13b_zoo": decode_13b_zoo,
    "mixed_iteration": mixed_iteration,
}


def by_name(name: str, **kw) -> Workload:
    return WORKLOADS[name](**kw)


def stacked_factors(w: Workload, ids: Sequence[int], p: int = 0) -> List[Tuple[np.ndarray, np.ndarray]]:
    """[(At_p, B_p)] for ``ids`` at projection ``p`` (views into the cached factors)."""
    out = []
    for a in ids:
        At, B = w.factors(int(a))
        out.append((At[p], B[p]))
    return out

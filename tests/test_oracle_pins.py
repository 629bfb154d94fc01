"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these re-types the oracle's formula and calls that a check.  Each compares the
oracle with something independent of it:

  * ``pin_half_decode``      -- all 65536 fp16 bit patterns against numpy's conversion
  * ``pin_golden``           -- hand-derived closed-form cases in tests/golden/
  * ``pin_merged_weight``    -- brute force with the merged weight W + s*A*B (the rejected
                                alternative the explainer page describes under "Prior
                                limits"): x(W + sAB) == xW + s*xAB, exact on integer inputs
  * ``pin_exact_rational``   -- pure-Python Fraction arithmetic on tiny random fp16 inputs
  * ``pin_grouped_blas``     -- numpy fp64 BLAS, tokens grouped by adapter: X_a A_a B_a
  * ``pin_zero_B``           -- B = 0 leaves y0 unchanged, bit for bit
  * ``pin_base_only``        -- index -1 leaves y0 unchanged
  * ``pin_invariances``      -- token order and adapter numbering do not change results
  * ``pin_projection_select``-- grouped numpy BLAS on projection 2 of a 3-projection
                                workload: the projection's own x, y0, At and B are used
  * ``pin_tolerance_mask``   -- the parity bound |got - ref| <= atol + rtol |ref| on
                                hand-worked values on both sides of it (negative refs,
                                got below and above ref, zero ref, NaN)

``test_mutants_are_caught`` plants mistakes in a copy of the oracle's C source (dropped
scaling, wrong sign, transposed operand, dropped term, wrong token, ...), compiles each
copy, and checks that the pins above reject every one of them.
``test_python_mutants_are_caught`` does the same for the Python side of the oracle
(projection selection, the tolerance mask).
"""
import ctypes
import json
import os
import shutil
import subprocess
import tempfile
from fractions import Fraction

import numpy as np
import pytest

import oracle
from rank_delta_paged_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f16(a):
    return np.asarray(a, dtype=np.float16)


# --------------------------------------------------------------------------- pins

def pin_half_decode():
    bits = np.arange(1 << 16, dtype=np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def pin_golden():
    for name in sorted(os.listdir(GOLDEN)):
        if not name.endswith(".json"):
            continue
        g = json.load(open(os.path.join(GOLDEN, name)))
        factors = [(_f16(At), _f16(B)) for At, B in zip(g["At"], g["B"])]
        ref = oracle.lora_delta(_f16(g["x"]), _f16(g["y0"]), np.array(g["idx"], np.int32),
                                np.array(g["ranks"]), np.array(g["scaling"]), factors)
        assert np.array_equal(ref, np.array(g["expected"], dtype=np.float64)), name


def pin_merged_weight():
    rng = np.random.default_rng(1234)
    d, T = 16, 6
    for r in (1, 2, 4, 8):
        s = 16.0 / r
        # integer inputs: every product and sum is exact in fp64 and in fp16
        x = rng.integers(-3, 4, size=(T, d)).astype(np.float16)
        Wb = rng.integers(-2, 3, size=(d, d)).astype(np.float64)
        A = rng.integers(-1, 2, size=(d, r)).astype(np.float16)
        B = rng.integers(-1, 2, size=(r, d)).astype(np.float16)
        y0 = (x.astype(np.float64) @ Wb).astype(np.float16)      # exact: |xW| <= 96
        merged = Wb + s * (A.astype(np.float64) @ B.astype(np.float64))
        want = x.astype(np.float64) @ merged
        ref = oracle.lora_delta(x, y0, np.zeros(T, np.int32), np.array([r]), np.array([s]),
                                [(A.T.copy(), B)])
        assert np.array_equal(ref, want), r
        # general fp16 values: agreement to fp64 rounding
        x = rng.standard_normal((T, d)).astype(np.float16)
        A = (rng.random((d, r)) - 0.5).astype(np.float16)
        B = (0.02 * rng.standard_normal((r, d))).astype(np.float16)
        y0 = rng.standard_normal((T, d)).astype(np.float16)
        merged_delta = s * (A.astype(np.float64) @ B.astype(np.float64))
        want = y0.astype(np.float64) + x.astype(np.float64) @ merged_delta
        ref = oracle.lora_delta(x, y0, np.zeros(T, np.int32), np.array([r]), np.array([s]),
                                [(A.T.copy(), B)])
        np.testing.assert_allclose(ref, want, rtol=1e-12, atol=1e-13)


def pin_exact_rational():
    rng = np.random.default_rng(99)
    d, T = 6, 5
    ranks = np.array([1, 3, 2])
    scal = np.array([16.0, 16.0 / 3.0, 8.0])
    facs = []
    for r in ranks:
        At = (rng.standard_normal((r, d)) * 0.3).astype(np.float16)
        B = (rng.standard_normal((r, d)) * 0.05).astype(np.float16)
        facs.append((At, B))
    x = rng.standard_normal((T, d)).astype(np.float16)
    y0 = rng.standard_normal((T, d)).astype(np.float16)
    idx = np.array([2, 0, -1, 1, 2], np.int32)
    ref = oracle.lora_delta(x, y0, idx, ranks, scal, facs)
    F = lambda v: Fraction(float(v))
    for t in range(T):
        a = int(idx[t])
        for n in range(d):
            exact = F(y0[t, n])
            if a >= 0:
                At, B = facs[a]
                s = Fraction(scal[a])
                tot = Fraction(0)
                for j in range(int(ranks[a])):
                    u = sum((F(x[t, k]) * F(At[j, k]) for k in range(d)), Fraction(0))
                    tot += u * F(B[j, n])
                exact += s * tot
            err = abs(Fraction(float(ref[t, n])) - exact)
            assert err <= Fraction(1, 10**12) * (1 + abs(exact)), (t, n, float(err))


def pin_grouped_blas():
    w = W.tiny_decode(seed=3)
    x, y0 = w.x(), w.y0()
    ref = oracle.workload_reference(w)
    want = y0.astype(np.float64).copy()
    for a in np.unique(w.token_adapter_idx):
        rows = np.nonzero(w.token_adapter_idx == a)[0]
        At, B = w.factors(int(a))
        X = x[rows].astype(np.float64)
        want[rows] += float(w.scaling()[a]) * (X @ At[0].T.astype(np.float64)) @ B[0].astype(np.float64)
    np.testing.assert_allclose(ref, want, rtol=1e-12, atol=1e-12)


def pin_zero_B():
    w = W.tiny_decode(seed=5)
    factors = []
    for a in range(w.n_adapters):
        At, B = w.factors(a)
        factors.append((At[0], np.zeros_like(B[0])))
    y0 = w.y0()
    ref = oracle.lora_delta(w.x(), y0, w.token_adapter_idx, w.ranks, w.scaling(), factors)
    assert np.array_equal(ref, y0.astype(np.float64))


def pin_base_only():
    w = W.tiny_decode(seed=6)
    idx = w.token_adapter_idx.copy()
    idx[::2] = -1
    y0 = w.y0()
    factors = [(w.factors(a)[0][0], w.factors(a)[1][0]) for a in range(w.n_adapters)]
    ref = oracle.lora_delta(w.x(), y0, idx, w.ranks, w.scaling(), factors)
    assert np.array_equal(ref[::2], y0[::2].astype(np.float64))
    assert not np.array_equal(ref[1::2], y0[1::2].astype(np.float64))


def pin_invariances():
    w = W.tiny_decode(seed=7, T=24)
    x, y0, idx = w.x(), w.y0(), w.token_adapter_idx
    factors = [(w.factors(a)[0][0], w.factors(a)[1][0]) for a in range(w.n_adapters)]
    ref = oracle.lora_delta(x, y0, idx, w.ranks, w.scaling(), factors)
    perm = np.random.default_rng(1).permutation(w.T)
    ref_p = oracle.lora_delta(x[perm], y0[perm], idx[perm], w.ranks, w.scaling(), factors)
    assert np.array_equal(ref_p, ref[perm])
    relabel = np.array([2, 0, 3, 1])           # old id a -> new id relabel[a]
    inv = np.argsort(relabel)
    ref_r = oracle.lora_delta(x, y0, relabel[idx].astype(np.int32), w.ranks[inv],
                              w.scaling()[inv], [factors[i] for i in inv])
    assert np.array_equal(ref_r, ref)


def pin_projection_select():
    base = W.tiny_decode(seed=9, T=12)
    w = W.Workload("tiny_3proj", base.hidden, 3, base.ranks, base.token_adapter_idx, None,
                   num_pages=3 * base.num_pages, kv_pages=0, shuffle_seed=5, seed=21)
    p = 2
    x, y0 = w.x(p), w.y0(p)
    # the projections really differ, so a wrong projection cannot agree by accident
    assert not np.array_equal(x, w.x(0)) and not np.array_equal(y0, w.y0(0))
    want = y0.astype(np.float64).copy()
    for a in np.unique(w.token_adapter_idx):
        if a < 0:
            continue
        rows = np.nonzero(w.token_adapter_idx == a)[0]
        At, B = w.factors(int(a))
        assert not np.array_equal(At[p], At[0])
        X = x[rows].astype(np.float64)
        want[rows] += float(w.scaling()[a]) * (X @ At[p].T.astype(np.float64)) @ B[p].astype(np.float64)
    np.testing.assert_allclose(oracle.workload_reference(w, p=p), want, rtol=1e-12, atol=1e-12)


def pin_tolerance_mask():
    # bound = 1e-3 + 1e-2 |ref|: 0.011, 0.021, 0.001, 0.006, 1.001, 0.011
    ref = np.array([1.0, -2.0, 0.0, -0.5, 100.0, -1.0])
    bound = np.array([0.011, 0.021, 0.001, 0.006, 1.001, 0.011])
    cases = [
        (ref + 0.9 * bound, [True] * 6),     # inside, above ref
        (ref - 0.9 * bound, [True] * 6),     # inside, below ref
        (ref + 1.1 * bound, [False] * 6),    # outside, above ref
        (ref - 1.1 * bound, [False] * 6),    # outside, below ref
        # a got of larger magnitude than ref, just inside the bound
        (np.array([1.0105, -2.0205, 0.0009, -0.5059, 100.999, -1.0108]), [True] * 6),
        # a got of smaller magnitude than ref, just inside the bound (a bound taken on |got|
        # would reject four of these); 0.0011 from a zero ref is outside
        (np.array([0.9895, -1.9792, -0.0011, -0.49405, 99.005, -0.98905]),
         [True, True, False, True, True, True]),
        (np.array([np.nan, -2.0, 0.0, np.inf, 100.0, -1.0]), [False, True, True, False, True, True]),
    ]
    for got, want in cases:
        mask = oracle.within_tolerance(got.astype(np.float64), ref, 1e-3, 1e-2)
        assert mask.tolist() == want, (got.tolist(), mask.tolist(), want)


PINS = [pin_half_decode, pin_golden, pin_merged_weight, pin_exact_rational,
        pin_grouped_blas, pin_zero_B, pin_base_only, pin_invariances,
        pin_projection_select, pin_tolerance_mask]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


# ------------------------------------------------------------ planted mistakes

MUTANTS = {
    "drop_scaling": ("o[n] += s * acc;", "o[n] += acc;"),
    "wrong_sign": ("o[n] += s * acc;", "o[n] -= s * acc;"),
    "transpose_At": ("slora_oracle_half_to_double(arow[k]);",
                     "slora_oracle_half_to_double(At[a][(size_t)k * (size_t)r + j]);"),
    "transpose_B": ("B[a][(size_t)j * (size_t)d + n]", "B[a][(size_t)n * (size_t)r + j]"),
    "drop_first_rank_term": ("for (int32_t j = 0; j < r; ++j)\n                acc += u[j]",
                             "for (int32_t j = 1; j < r; ++j)\n                acc += u[j]"),
    "drop_last_k_term": ("for (int32_t k = 0; k < d; ++k)", "for (int32_t k = 0; k < d - 1; ++k)"),
    "no_base": ("o[n] = slora_oracle_half_to_double(yt[n]);", "o[n] = 0.0;"),
    "wrong_token_x": ("slora_oracle_half_to_double(xt[k])", "slora_oracle_half_to_double(x[k])"),
    "half_exponent_bias": ("e - 25", "e - 24"),
    "subnormal_scale": ("(double)m, -24", "(double)m, -25"),
}


def _build_mutant(tmp, name, old, new):
    src = open(oracle._SRC).read()
    assert old in src, name
    src = src.replace(old, new, 1)
    cpath = os.path.join(tmp, f"{name}.c")
    open(cpath, "w").write(src)
    so = os.path.join(tmp, f"lib{name}.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", so, cpath,
                    "-lm"], check=True)
    return so


def _pins_pass():
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            return False
    return True


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
def test_mutants_are_caught():
    oracle._load()
    real = oracle._lib
    tmp = tempfile.mkdtemp(prefix="oracle_mutants_")
    survived = []
    try:
        for name, (old, new) in MUTANTS.items():
            lib = ctypes.CDLL(_build_mutant(tmp, name, old, new))
            for fn in ("slora_oracle_half_to_double", "slora_oracle_threads", "slora_oracle_delta"):
                getattr(lib, fn).restype = getattr(real, fn).restype
                getattr(lib, fn).argtypes = getattr(real, fn).argtypes
            oracle._lib = lib
            if _pins_pass():
                survived.append(name)
    finally:
        oracle._lib = real
        shutil.rmtree(tmp, ignore_errors=True)
    assert not survived, f"pins missed planted mistakes: {survived}"


# Mistakes planted in the Python side of the oracle (projection selection and the parity
# bound), each applied to a copy of the function's source in the module's namespace.
PY_MUTANTS = {
    "factor_of_projection_0": ("workload_reference", "factors[a] = (At[p], B[p])",
                               "factors[a] = (At[0], B[p])"),
    "B_of_projection_0": ("workload_reference", "factors[a] = (At[p], B[p])",
                          "factors[a] = (At[p], B[0])"),
    "x_of_projection_0": ("workload_reference", "x = w.x(p) if x is None else x",
                          "x = w.x(0) if x is None else x"),
    "rtol_times_got": ("within_tolerance", "rtol * np.abs(ref)", "rtol * np.abs(got)"),
    "dropped_abs": ("within_tolerance", "np.abs(got.astype(np.float64) - ref)",
                    "(got.astype(np.float64) - ref)"),
    "rtol_dropped": ("within_tolerance", "atol + rtol * np.abs(ref)", "atol + np.abs(ref) * 0"),
}


def test_python_mutants_are_caught():
    import inspect
    import textwrap
    survived = []
    for name, (fn, old, new) in PY_MUTANTS.items():
        real = getattr(oracle, fn)
        src = textwrap.dedent(inspect.getsource(real))
        assert old in src, name
        ns = dict(vars(oracle))
        exec(compile(src.replace(old, new, 1), f"<mutant {name}>", "exec"), ns)
        setattr(oracle, fn, ns[fn])
        try:
            if _pins_pass():
                survived.append(name)
        finally:
            setattr(oracle, fn, real)
    assert not survived, f"pins missed planted mistakes: {survived}"

"""CPU oracle for the paged heterogeneous-rank LoRA delta -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import this package.  The product (``rank_delta_paged_gb300``) never
imports it, and it never imports the product: the two share no code.  The only module
both sides use is ``rank_delta_paged_gb300.workloads``, which draws seeded inputs and
holds none of the delta's arithmetic.

The arithmetic lives in ``slora_oracle.c`` (plain C, fp64, one OpenMP loop over tokens),
built here with gcc into ``oracle/_build/libslora_oracle.so`` and called through ctypes.
What it computes, per token t with adapter a (S-LoRA: Serving Thousands of Concurrent
LoRA Adapters (explainer), "What this paper explains" and "How to read the paper";
S-LoRA: Multiplexing Thousands of Fine-Tuned Adapters on a Single GPU, section 2
pseudocode)::

    ref[t] = y0[t] + s_a * (x[t] @ A_a) @ B_a          (A_a = At_a.T)

Every function is pinned by ``tests/test_oracle_pins.py`` against things other than
itself: exhaustive fp16 decoding against numpy, merged-weight brute force, exact
rational arithmetic, grouped BLAS, invariants and hand-derived golden cases.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "slora_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libslora_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.slora_oracle_half_to_double.restype = ctypes.c_double
            lib.slora_oracle_half_to_double.argtypes = [ctypes.c_uint16]
            lib.slora_oracle_threads.restype = ctypes.c_int
            lib.slora_oracle_threads.argtypes = []
            lib.slora_oracle_set_threads.restype = None
            lib.slora_oracle_set_threads.argtypes = [ctypes.c_int]
            P = ctypes.c_void_p
            lib.slora_oracle_delta.restype = ctypes.c_int
            lib.slora_oracle_delta.argtypes = [ctypes.c_int32, ctypes.c_int32, P, P, P,
                                               ctypes.c_int32, P, P, P, P,
                                               ctypes.c_int64, P, P]
            _lib = lib
    return _lib


def threads() -> int:
    """OpenMP threads the oracle runs on (set OMP_NUM_THREADS before the first call)."""
    return int(_load().slora_oracle_threads())


def set_threads(n: int) -> None:
    """Run later oracle calls on n OpenMP threads (timing only; results do not change)."""
    _load().slora_oracle_set_threads(int(n))


def half_to_double(bits: int) -> float:
    return float(_load().slora_oracle_half_to_double(int(bits) & 0xFFFF))


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def lora_delta(x: np.ndarray, y0: np.ndarray, idx: np.ndarray, ranks: np.ndarray,
               scaling: np.ndarray, factors: Sequence, sel: Optional[np.ndarray] = None
               ) -> np.ndarray:
    """fp64 reference outputs.

    x, y0    fp16 [T][d];  idx int32 [T] (-1 = base only)
    ranks    int [n_adapters];  scaling float [n_adapters]
    factors  sequence indexed by adapter id: (At [r][d] fp16, B [r][d] fp16), or None
             for adapters no selected token uses
    sel      int32 token indices to compute (None = all tokens)
    Returns float64 [len(sel) or T][d].
    """
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float16)
    y0 = np.ascontiguousarray(y0, dtype=np.float16)
    T, d = x.shape
    assert y0.shape == (T, d)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    assert idx.shape == (T,)
    n_ad = len(factors)
    ranks_c = np.ascontiguousarray(ranks[:n_ad], dtype=np.int32)
    scal_c = np.ascontiguousarray(scaling[:n_ad], dtype=np.float64)
    keep = []
    At_p = (ctypes.c_void_p * max(n_ad, 1))()
    B_p = (ctypes.c_void_p * max(n_ad, 1))()
    for a, f in enumerate(factors):
        if f is None:
            continue
        At, B = f
        At = np.ascontiguousarray(At, dtype=np.float16)
        B = np.ascontiguousarray(B, dtype=np.float16)
        assert At.shape == (int(ranks_c[a]), d) and B.shape == At.shape, (a, At.shape)
        keep += [At, B]
        At_p[a] = _ptr(At)
        B_p[a] = _ptr(B)
    if sel is None:
        sel_c = None
        n_sel = T
    else:
        sel_c = np.ascontiguousarray(sel, dtype=np.int32)
        n_sel = int(sel_c.shape[0])
    out = np.empty((n_sel, d), dtype=np.float64)
    rc = lib.slora_oracle_delta(T, d, _ptr(x), _ptr(y0), _ptr(idx), n_ad, _ptr(ranks_c),
                                _ptr(scal_c), ctypes.cast(At_p, ctypes.c_void_p),
                                ctypes.cast(B_p, ctypes.c_void_p), n_sel,
                                None if sel_c is None else _ptr(sel_c), _ptr(out))
    if rc != 0:
        raise ValueError("oracle: adapter index out of range or missing factors")
    return out


def workload_reference(w, p: int = 0, sel: Optional[np.ndarray] = None,
                       x: Optional[np.ndarray] = None, y0: Optional[np.ndarray] = None
                       ) -> np.ndarray:
    """Reference outputs of projection ``p`` of a ``workloads.Workload`` (factors read
    from the workload's host arrays, never from a device pool)."""
    x = w.x(p) if x is None else x
    y0 = w.y0(p) if y0 is None else y0
    idx = w.token_adapter_idx
    toks = np.arange(w.T) if sel is None else np.asarray(sel)
    need = set(int(a) for a in idx[toks] if a >= 0)
    factors = [None] * w.n_adapters
    for a in need:
        At, B = w.factors(a)
        factors[a] = (At[p], B[p])
    return lora_delta(x, y0, idx, w.ranks, w.scaling(), factors, sel)


def within_tolerance(got: np.ndarray, ref: np.ndarray, atol: float = 1e-3,
                     rtol: float = 1e-2) -> np.ndarray:
    """Element mask of |got - ref| <= atol + rtol * |ref|."""
    return np.abs(got.astype(np.float64) - ref) <= atol + rtol * np.abs(ref)

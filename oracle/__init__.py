"""CPU oracle for exact row-wise FP32 Top-K (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The product path (the CUDA
library and its binding) never imports, links or executes anything here, and
this package never imports the product.

Two oracles are exposed, both implemented in ``exact_topk_oracle.cpp``:

* :func:`topk_rows` -- the plain definition of the operator ("Sample-Guided
  Exact Top-K Selection for Long-Context Sparse Attention", section 2.1
  "Operator contract"): per row the K largest valid scores, found with
  ``std::nth_element`` on the FP32 total-order key; rows with ``L <= K``
  return every valid index followed by -1.
* :func:`method_trace` -- the three-phase sample-guided method written out
  step by step (sections 4.2-4.4, eqs. 11-25) with its per-row trace: route
  (Table 2), tau0, tau1, C(tau0), C(tau1), tau*, |E0|, |Q0|.

Parity of every function here is pinned in ``tests/test_oracle_pins.py``
against brute force, numpy's sort and binary16 cast, closed forms and
hand-computed fixtures under ``tests/golden/``.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import build_oracle

ROUTE_PAD = 0
ROUTE_PRIMARY = 1
ROUTE_BAND = 2
ROUTE_EXACT_AFTER_BAND = 3
ROUTE_EXACT_NO_BAND = 4
ROUTE_DIRECT_EXACT = 5
ROUTE_GUESS = 6
ROUTE_GUESS_EXACT = 7

ROUTE_NAMES = {
    ROUTE_PAD: "pad",
    ROUTE_PRIMARY: "primary",
    ROUTE_BAND: "band",
    ROUTE_EXACT_AFTER_BAND: "exact_after_band",
    ROUTE_EXACT_NO_BAND: "exact_no_band",
    ROUTE_DIRECT_EXACT: "direct_exact",
    ROUTE_GUESS: "guess",
    ROUTE_GUESS_EXACT: "guess_exact",
}

TRACE_FIELDS = ("route", "tau0", "tau1", "c0", "c1", "tau_star", "e0", "q0")

_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    path = build_oracle()
    lib = ctypes.CDLL(path)
    i64, i32, p = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    lib.oracle_topk_rows.argtypes = [p, i64, i64, i64, p, i64, i32, p, i32]
    lib.oracle_topk_rows.restype = i32
    lib.oracle_method_trace.argtypes = [p, i64, i64, i64, p, i64, i32, i32, i32, i32, i32, i32, i32,
                                        i32, p, p, p, i32]
    lib.oracle_method_trace.restype = i32
    lib.oracle_f16_bits.argtypes = [ctypes.c_float]
    lib.oracle_f16_bits.restype = ctypes.c_uint16
    lib.oracle_coarse_bin.argtypes = [ctypes.c_float]
    lib.oracle_coarse_bin.restype = i32
    lib.oracle_desc32.argtypes = [ctypes.c_float]
    lib.oracle_desc32.restype = ctypes.c_uint32
    lib.oracle_cutoff_for_bin.argtypes = [i32]
    lib.oracle_cutoff_for_bin.restype = ctypes.c_uint32
    lib.oracle_view_phase.argtypes = [i64, i32]
    lib.oracle_view_phase.restype = i32
    lib.oracle_f16_bits_array.argtypes = [p, i64, p]
    lib.oracle_f16_bits_array.restype = None
    lib.oracle_coarse_bin_array.argtypes = [p, i64, p]
    lib.oracle_coarse_bin_array.restype = None
    lib.oracle_hardware_threads.argtypes = []
    lib.oracle_hardware_threads.restype = i32
    _lib = lib
    return lib


def hardware_threads() -> int:
    return int(_load().oracle_hardware_threads())


def _threads(nthreads):
    if nthreads is None:
        return hardware_threads()
    return max(1, int(nthreads))


def _matrix(X):
    X = np.asarray(X)
    if X.dtype != np.float32:
        raise TypeError("scores must be float32")
    if X.ndim != 2:
        raise ValueError("scores must be [M, N]")
    if X.shape[0] <= 1 or X.strides[1] != 4 or X.strides[0] % 4 or X.strides[0] < 4 * X.shape[1]:
        X = np.ascontiguousarray(X)
        return X, X.shape[1]
    return X, X.strides[0] // 4


def topk_rows(X, ke, K, M_live=None, out=None, nthreads=None):
    """Per-row exact Top-K by definition; returns ``out`` [M, K] int32.

    Rows ``r >= M_live`` of ``out`` are not written (a fresh ``out`` is filled
    with the canary -7 there)."""
    X, pitch = _matrix(X)
    M, N = X.shape
    ke = np.ascontiguousarray(ke, dtype=np.int32)
    if ke.shape != (M,):
        raise ValueError("ke must be [M]")
    if M_live is None:
        M_live = M
    if out is None:
        out = np.full((M, K), -7, dtype=np.int32)
    rc = _load().oracle_topk_rows(X.ctypes.data, M, N, pitch, ke.ctypes.data, int(M_live), int(K),
                                  out.ctypes.data, _threads(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_topk_rows failed ({rc})")
    return out


def method_trace(X, ke, K, s, dual, rho0=(3, 2), rho1=(7, 4), sampled=True, guess=None,
                 M_live=None, nthreads=None):
    """The three-phase method with its per-row trace.

    Returns ``(out [M, K] int32, trace [M, 8] int32)``; trace columns are
    :data:`TRACE_FIELDS`, -1 where a field was not computed on that route."""
    X, pitch = _matrix(X)
    M, N = X.shape
    ke = np.ascontiguousarray(ke, dtype=np.int32)
    if M_live is None:
        M_live = M
    out = np.full((M, K), -7, dtype=np.int32)
    trace = np.full((M, len(TRACE_FIELDS)), -7, dtype=np.int32)
    gptr = None
    if guess is not None:
        guess = np.ascontiguousarray(guess, dtype=np.int32)
        if guess.shape != (M, K):
            raise ValueError("guess must be [M, K]")
        gptr = guess.ctypes.data
    rc = _load().oracle_method_trace(X.ctypes.data, M, N, pitch, ke.ctypes.data, int(M_live), int(K),
                                     int(s), int(bool(dual)), int(rho0[0]), int(rho0[1]),
                                     int(rho1[0]), int(rho1[1]), int(bool(sampled)), gptr,
                                     out.ctypes.data, trace.ctypes.data, _threads(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_method_trace failed ({rc})")
    return out, trace


def f16_bits(x: float) -> int:
    return int(_load().oracle_f16_bits(float(x)))


def f16_bits_array(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_f16_bits_array(x.ctypes.data, x.size, out.ctypes.data)
    return out


def coarse_bin(x: float) -> int:
    return int(_load().oracle_coarse_bin(float(x)))


def coarse_bin_array(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.empty(x.shape, dtype=np.int32)
    _load().oracle_coarse_bin_array(x.ctypes.data, x.size, out.ctypes.data)
    return out


def desc32(x: float) -> int:
    return int(_load().oracle_desc32(float(x)))


def cutoff_for_bin(tau: int) -> int:
    return int(_load().oracle_cutoff_for_bin(int(tau)))


def view_phase(r: int, s: int) -> int:
    return int(_load().oracle_view_phase(int(r), int(s)))


def library_path() -> str:
    return os.path.abspath(build_oracle())

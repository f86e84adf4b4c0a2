"""fp64 CPU oracle for the symbolic kernel reductions -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and shares
no code with it.  The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over
rows); this module compiles it with gcc and wraps it with ctypes.

Functions (each follows the passage cited in ``oracle.c``):

* ``gauss_sum(x, y, b, sigma)``   -> (a, S)   Sum reduction and its tolerance scale
* ``gauss_lse(x, y, w, sigma)``   -> L        LogSumExp with additive log-weights
* ``gauss_grad_x(x, y, b, g, sigma)`` -> (gx, G)  x-gradient of sum(g * a) and its scale
* ``gauss_grad_y(x, y, b, g, sigma)`` -> (gy, G)  y-gradient of sum(g * a) and its scale
* ``gauss_grad_b(x, y, g, sigma)``    -> (gb, S)  b-gradient (transposed product) and its scale
* ``kernel_sum(x, y, b, sigma, kernel)`` -> (a, S)  Sum with a Gaussian, Laplace, Cauchy or
  inverse-multiquadric kernel
* ``kernel_maxmin(x, y, b, sigma, kernel, "max"|"min")`` -> (val, idx, second)  Max / Min of
  k b over j with the lowest attaining index and the runner-up value
* ``kernel_ranges(x, y, b, sigma, kernel, "sum"|"max"|"min", ranges_i, slices_i, redranges_j)``
  block-sparse Sum / Max / Min over per-cluster column ranges
* ``knn(x, y, K)``                -> (idx, dist, next)  K-min by (distance, index)

Inputs may be float32 or float64 arrays; they are converted to float64 (exact for
float32).  b, w, g accept shape (N,) / (M,) for E = 1.

Parity: every function here is pinned by the tests in ``tests/test_oracle_pins.py``
(closed forms, invariants, library special cases, finite differences).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_dp = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def build(src: str = _SRC, out: str = _LIB, extra_flags=()) -> str:
    """Compile ``oracle.c`` into a shared library with gcc (OpenMP, no fast-math)."""
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-fno-fast-math", "-ffp-contract=off", *extra_flags, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _as2d(a, rows, name):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if a.ndim == 1:
        a = a.reshape(rows, 1) if rows else a.reshape(0, 1)
    if a.ndim != 2 or a.shape[0] != rows:
        raise ValueError(f"{name}: expected {rows} rows, got shape {a.shape}")
    return a


def _ptr(a):
    return a.ctypes.data_as(_dp)


class Oracle:
    """ctypes handle on one compiled oracle library (the real one, or a test mutant)."""

    def __init__(self, path: str = _LIB):
        if not os.path.exists(path):
            raise FileNotFoundError(f"oracle library not built: {path} (call oracle.build())")
        lib = ctypes.CDLL(path)
        lib.oracle_gauss_sum.argtypes = [_dp, _dp, _dp, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_double, _dp, _dp]
        lib.oracle_gauss_lse.argtypes = [_dp, _dp, _dp, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_double, _dp]
        lib.oracle_gauss_grad_x.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_double, _dp, _dp]
        lib.oracle_gauss_grad_y.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_double, _dp, _dp]
        lib.oracle_gauss_grad_b.argtypes = [_dp, _dp, _dp, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_double, _dp, _dp]
        lib.oracle_kernel_sum.argtypes = [_dp, _dp, _dp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_double, ctypes.c_int, _dp, _dp]
        lib.oracle_kernel_maxmin.argtypes = [_dp, _dp, _dp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int, _dp,
                                             _i64p, _dp]
        lib.oracle_kernel_ranges.argtypes = [_dp, _dp, _dp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int64, _i64p, _i64p, _i64p, _dp, _dp, _i64p, _dp]
        lib.oracle_knn.argtypes = [_dp, _dp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                   ctypes.c_int, _i64p, _dp, _dp]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        self._lib = lib
        self.path = path

    # -- threads ---------------------------------------------------------
    def num_threads(self) -> int:
        return int(self._lib.oracle_num_threads())

    def set_num_threads(self, n: int) -> None:
        self._lib.oracle_set_num_threads(int(n))

    # -- shapes ----------------------------------------------------------
    @staticmethod
    def _points(x, y):
        x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
        y = np.ascontiguousarray(np.asarray(y, dtype=np.float64))
        if x.ndim != 2 or y.ndim != 2 or x.shape[1] != y.shape[1]:
            raise ValueError(f"x, y must be (M, D) and (N, D); got {x.shape}, {y.shape}")
        return x, y

    # -- reductions ------------------------------------------------------
    def gauss_sum(self, x, y, b, sigma):
        x, y = self._points(x, y)
        M, D = x.shape
        N = y.shape[0]
        b = _as2d(b, N, "b")
        E = b.shape[1]
        a = np.empty((M, E))
        S = np.empty((M, E))
        self._lib.oracle_gauss_sum(_ptr(x), _ptr(y), _ptr(b), M, N, D, E, float(sigma),
                                   _ptr(a), _ptr(S))
        return a, S

    def gauss_lse(self, x, y, w, sigma):
        x, y = self._points(x, y)
        M, D = x.shape
        N = y.shape[0]
        w = _as2d(w, N, "w")
        E = w.shape[1]
        L = np.empty((M, E))
        self._lib.oracle_gauss_lse(_ptr(x), _ptr(y), _ptr(w), M, N, D, E, float(sigma), _ptr(L))
        return L

    def gauss_grad_x(self, x, y, b, g, sigma):
        x, y = self._points(x, y)
        M, D = x.shape
        N = y.shape[0]
        b = _as2d(b, N, "b")
        E = b.shape[1]
        g = _as2d(g, M, "g")
        if g.shape[1] != E:
            raise ValueError(f"g must have E={E} columns, got {g.shape}")
        gx = np.empty((M, D))
        G = np.empty((M, D))
        self._lib.oracle_gauss_grad_x(_ptr(x), _ptr(y), _ptr(b), _ptr(g), M, N, D, E,
                                      float(sigma), _ptr(gx), _ptr(G))
        return gx, G

    def gauss_grad_y(self, x, y, b, g, sigma):
        x, y = self._points(x, y)
        M, D = x.shape
        N = y.shape[0]
        b = _as2d(b, N, "b")
        E = b.shape[1]
        g = _as2d(g, M, "g")
        if g.shape[1] != E:
            raise ValueError(f"g must have E={E} columns, got {g.shape}")
        gy = np.empty((N, D))
        G = np.empty((N, D))
        self._lib.oracle_gauss_grad_y(_ptr(x), _ptr(y), _ptr(b), _ptr(g), M, N, D, E,
                                      float(sigma), _ptr(gy), _ptr(G))
        return gy, G

    def gauss_grad_b(self, x, y, g, sigma):
        x, y = self._points(x, y)
        M, D = x.shape
        N = y.shape[0]
        g = _as2d(g, M, "g")
        E = g.shape[1]
        gb = np.empty((N, E))
        S = np.empty((N, E))
        self._lib.oracle_gauss_grad_b(_ptr(x), _ptr(y), _ptr(g), M, N, D, E, float(sigma),
                                      _ptr(gb), _ptr(S))
        return gb, S

    def kernel_sum(self, x, y, b, sigma, kernel):
        x, y = self._points(x, y)
        M, D = x.shape
        N = y.shape[0]
        b = _as2d(b, N, "b")
        E = b.shape[1]
        a = np.empty((M, E))
        S = np.empty((M, E))
        self._lib.oracle_kernel_sum(_ptr(x), _ptr(y), _ptr(b), M, N, D, E, float(sigma), KERNELS[kernel],
                                    _ptr(a), _ptr(S))
        return a, S

    def kernel_maxmin(self, x, y, b, sigma, kernel, reduction):
        x, y = self._points(x, y)
        M, D = x.shape
        N = y.shape[0]
        b = _as2d(b, N, "b")
        E = b.shape[1]
        sense = {"max": 1, "min": -1}[reduction]
        val = np.empty((M, E))
        idx = np.empty((M, E), dtype=np.int64)
        second = np.empty((M, E))
        self._lib.oracle_kernel_maxmin(_ptr(x), _ptr(y), _ptr(b), M, N, D, E, float(sigma), KERNELS[kernel],
                                       sense, _ptr(val), idx.ctypes.data_as(_i64p), _ptr(second))
        return val, idx, second

    def kernel_ranges(self, x, y, b, sigma, kernel, reduction, ranges_i, slices_i, redranges_j):
        """Block-sparse Sum / Max / Min.  ranges_i (nc, 2) row clusters [start, end),
        slices_i (nc,) cumulative ends into redranges_j (nr, 2) column ranges [start, end).
        Returns (a, S) for "sum", (val, idx, second) for "max" / "min"."""
        x, y = self._points(x, y)
        M, D = x.shape
        N = y.shape[0]
        b = _as2d(b, N, "b")
        E = b.shape[1]
        ri = np.ascontiguousarray(np.asarray(ranges_i, dtype=np.int64).reshape(-1, 2))
        si = np.ascontiguousarray(np.asarray(slices_i, dtype=np.int64).reshape(-1))
        rj = np.ascontiguousarray(np.asarray(redranges_j, dtype=np.int64).reshape(-1, 2))
        if si.shape[0] != ri.shape[0]:
            raise ValueError("slices_i needs one entry per row cluster")
        red = {"sum": 0, "max": 1, "min": -1}[reduction]
        val = np.empty((M, E))
        scale = np.empty((M, E))
        idx = np.empty((M, E), dtype=np.int64)
        second = np.empty((M, E))
        p64 = lambda a: a.ctypes.data_as(_i64p)
        self._lib.oracle_kernel_ranges(_ptr(x), _ptr(y), _ptr(b), M, N, D, E, float(sigma), KERNELS[kernel], red,
                                       ri.shape[0], p64(ri), p64(si), p64(rj), _ptr(val), _ptr(scale), p64(idx),
                                       _ptr(second))
        if red == 0:
            return val, scale
        return val, idx, second

    def knn(self, x, y, K):
        x, y = self._points(x, y)
        M, D = x.shape
        N = y.shape[0]
        K = int(K)
        if K < 1:
            raise ValueError("K must be >= 1")
        idx = np.empty((M, K), dtype=np.int64)
        dist = np.empty((M, K))
        nxt = np.empty(M)
        self._lib.oracle_knn(_ptr(x), _ptr(y), M, N, D, K,
                             idx.ctypes.data_as(_i64p), _ptr(dist), _ptr(nxt))
        return idx, dist, nxt


# Radial kernels of oracle_kernel_sum / oracle_kernel_maxmin, by name.
KERNELS = {"gaussian": 0, "laplace": 1, "cauchy": 2, "imq": 3}

_default = None


def load(path: str = _LIB) -> Oracle:
    """The oracle compiled from ``oracle.c`` (built on first use if missing)."""
    global _default
    if path != _LIB:
        return Oracle(path)
    if _default is None:
        if not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            build()
        _default = Oracle(_LIB)
    return _default

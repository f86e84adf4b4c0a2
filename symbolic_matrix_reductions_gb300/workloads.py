"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers; it holds none of the reductions'
arithmetic, and both the CUDA path's tests and the oracle's tests take their
inputs from it.  Every array is float32, row-major, generated on the host with
NumPy's PCG64; each array has its own child stream spawned from the seed, so a
row subset or a size change in one array never changes another.

Workloads (the pages measure no public dataset; these stand in for them):

* ``gauss_small``  -- M=N=1000, D=3, E=1; x, y, b ~ N(0,1); sigma=1.  The D=3
  point clouds of the Gaussian matrix-vector benchmark ("Kernel Operations on the
  GPU...", §3, M = N points in dimension 3), at a size the oracle finishes at once.
* ``gauss_d3``     -- M=N=100000, D=3, E=1; x, y, b ~ N(0,1); sigma=0.5.
* ``gauss_d3_unit`` -- M=N=1000000, D=3, E=1; x, y ~ U[0,1]^3; b ~ U(0.1,1);
  sigma=0.1; the LogSumExp weight is w = log b.
* ``falkon_d50``   -- M=100000, N=10000000, D=50, E=1; x, y ~ N(0, I/50);
  b ~ N(0,1); sigma=1.  The tall kernel-vector product of the billion-scale
  GitHub issue ("Transparent interface for billion-scale matrices": N=1G,
  M=100k, D=50), with N scaled to 10^7.
* ``knn_d16``      -- M=N=1000000, D=16, K=10; 64 centres ~ N(0, I_16), labels
  uniform and independent for x and y, points = centre + 0.1 N(0, I_16).  The
  K-nearest-neighbour queries of the KeOps README.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    D: int
    E: int = 1
    sigma: float = 1.0
    K: int = 0
    seed: int = 0
    points: str = "normal"      # normal | unit_cube | normal_over_d | mixture
    weights: str = "normal"     # normal | uniform_0.1_1
    note: str = ""
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "gauss_small": Workload("gauss_small", 1000, 1000, 3, 1, 1.0, 0, 1001, "normal", "normal",
                            "Sum + grad of sum(a^2), M=N=1000, D=3"),
    "gauss_d3": Workload("gauss_d3", 100_000, 100_000, 3, 1, 0.5, 10, 1002, "normal", "normal",
                         "Sum + grad-x, M=N=1e5, D=3, sigma=0.5"),
    "gauss_d3_unit": Workload("gauss_d3_unit", 1_000_000, 1_000_000, 3, 1, 0.1, 0, 1003,
                              "unit_cube", "uniform_0.1_1",
                              "Sum and LogSumExp (w = log b), M=N=1e6, D=3, sigma=0.1"),
    "falkon_d50": Workload("falkon_d50", 100_000, 10_000_000, 50, 1, 1.0, 0, 1004,
                           "normal_over_d", "normal",
                           "tall product, M=1e5, N=1e7, D=50, split-j"),
    "knn_d16": Workload("knn_d16", 1_000_000, 1_000_000, 16, 1, 1.0, 10, 1005, "mixture", "normal",
                        "K-min K=10, M=N=1e6, D=16, 64-component mixture"),
}


def _streams(seed: int):
    """Independent child generators: x, y, weights, upstream gradient, mixture
    centres, x labels, y labels."""
    ss = np.random.SeedSequence(seed)
    return [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(7)]


def _points(rng, n, D, kind, centres=None, labels_rng=None):
    if kind == "normal":
        return rng.standard_normal((n, D), dtype=np.float32)
    if kind == "normal_over_d":
        return (rng.standard_normal((n, D), dtype=np.float32)
                * np.float32(1.0 / np.sqrt(D))).astype(np.float32)
    if kind == "unit_cube":
        return rng.random((n, D), dtype=np.float32)
    if kind == "mixture":
        lab = labels_rng.integers(0, centres.shape[0], size=n)
        pts = centres[lab] + np.float32(0.1) * rng.standard_normal((n, D), dtype=np.float32)
        return pts.astype(np.float32)
    raise ValueError(kind)


def generate(w: Workload | str, M: int | None = None, N: int | None = None,
             seed: int | None = None):
    """Draw the inputs of workload ``w`` (optionally resized to M x N).

    Returns a dict with float32 arrays ``x`` (M,D), ``y`` (N,D), ``b`` (N,E),
    ``g`` (M,E) (an upstream gradient ~ N(0,1), used where the pages leave it
    open), and for positive weights ``w_log`` (N,E) = log b, the LogSumExp
    weight.  Resizing keeps the distributions; it draws fresh numbers.
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    M = w.M if M is None else int(M)
    N = w.N if N is None else int(N)
    seed = w.seed if seed is None else int(seed)
    rx, ry, rb, rg, rc, lab_x, lab_y = _streams(seed)
    centres = None
    if w.points == "mixture":
        centres = rc.standard_normal((64, w.D), dtype=np.float32)
    x = _points(rx, M, w.D, w.points, centres, lab_x)
    y = _points(ry, N, w.D, w.points, centres, lab_y)
    if w.weights == "normal":
        b = rb.standard_normal((N, w.E), dtype=np.float32)
    elif w.weights == "uniform_0.1_1":
        b = (np.float32(0.1) + np.float32(0.9) * rb.random((N, w.E), dtype=np.float32)).astype(np.float32)
    else:
        raise ValueError(w.weights)
    g = rg.standard_normal((M, w.E), dtype=np.float32)
    out = {"x": x, "y": y, "b": b, "g": g, "sigma": float(w.sigma), "K": w.K}
    if w.weights == "uniform_0.1_1":
        out["w_log"] = np.log(b).astype(np.float32)
    return out


def row_subset(M: int, count: int, seed: int) -> np.ndarray:
    """A seeded sorted subset of ``count`` distinct row indices out of M."""
    rng = np.random.Generator(np.random.PCG64(seed))
    count = min(int(count), int(M))
    return np.sort(rng.choice(M, size=count, replace=False))

"""Pins for the fp64 oracle: facts fixed by the definitions, not by the oracle.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises ``AssertionError`` when the
oracle disagrees with something the mathematics fixes independently of it:
closed forms derived by hand (``tests/golden/closed_forms.json``), the Gaussian
integral, invariances, special cases that reduce to a library routine (SciPy's
distance matrix, NumPy's stable sort, a k-d tree), and central finite
differences of the (separately pinned) Sum reduction.  The list ``PINS`` is run
against the real oracle by ``test_oracle_pins.py`` and against deliberately
broken copies of it by ``test_oracle_mutants.py``.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "closed_forms.json")

_NS = {"exp": math.exp, "log": math.log, "sqrt": math.sqrt, "pi": math.pi, "inf": math.inf}


def _val(expr):
    if isinstance(expr, (int, float)):
        return float(expr)
    return float(eval(expr, {"__builtins__": {}}, _NS))  # hand-written closed forms only


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _close(a, b, rtol, atol=0.0, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    with np.errstate(invalid="ignore"):
        ok = (a == b) | (np.abs(a - b) <= atol + rtol * np.abs(b))
    assert ok.all(), f"{what}: {a[~ok][:4]} vs {b[~ok][:4]} (rtol {rtol}, atol {atol})"


# ---------------------------------------------------------------------------
# Sum reduction
# ---------------------------------------------------------------------------
def pin_sum_golden(orc):
    """Hand-derived values ('Kernel Operations on the GPU...', §1 target operation)."""
    for case in _golden()["sum"]:
        a, S = orc.gauss_sum(case["x"], case["y"], case["b"], case["sigma"])
        want = np.array([[_val(e) for e in row] for row in case["expect"]])
        _close(a, want, 1e-14, 1e-300, case["name"])


def pin_sum_single_point_identity(orc):
    """x_i = y_j with N = 1: the kernel is exactly 1, so a = b."""
    r = _rng(1)
    y = r.standard_normal((1, 5))
    b = r.standard_normal((1, 3))
    a, _ = orc.gauss_sum(y.copy(), y, b, 0.37)
    assert np.array_equal(a, b), (a, b)


def pin_sum_gaussian_integral_1d(orc):
    """Riemann sum on a fine uniform grid -> integral of exp(-t^2/sigma^2) = sigma sqrt(pi).

    Fixes the sigma convention and the sign of the exponent (a factor 2 in the
    denominator would give sigma sqrt(2 pi)).  For a Gaussian the uniform-grid
    sum converges faster than any power of h, so the fp64 result is exact to
    rounding."""
    sigma, h = 0.7, 0.05
    y = (-12.0 + h * np.arange(int(24 / h) + 1))[:, None]
    b = np.full((y.shape[0], 1), h)
    for x0 in (0.0, 0.3, -1.1):
        a, _ = orc.gauss_sum(np.array([[x0]]), y, b, sigma)
        _close(a[0, 0], sigma * math.sqrt(math.pi), 1e-12, 0, f"1-D integral at {x0}")


def pin_sum_gaussian_integral_3d(orc):
    """3-D tensor grid -> (sigma sqrt(pi))^3: every coordinate enters the distance."""
    sigma, h = 1.0, 0.2
    t = -6.0 + h * np.arange(int(12 / h) + 1)
    g = np.stack(np.meshgrid(t, t, t, indexing="ij"), -1).reshape(-1, 3)
    b = np.full((g.shape[0], 1), h ** 3)
    a, _ = orc.gauss_sum(np.array([[0.1, -0.2, 0.05]]), g, b, sigma)
    _close(a[0, 0], (sigma * math.sqrt(math.pi)) ** 3, 1e-10, 0, "3-D integral")


def pin_sum_bruteforce_scipy(orc):
    """Tiny inputs against SciPy's pairwise distance routine and a dense product."""
    from scipy.spatial.distance import cdist
    r = _rng(2)
    for (M, N, D, E, sigma) in [(7, 11, 3, 2, 0.9), (13, 5, 1, 1, 0.3), (4, 9, 6, 3, 2.5)]:
        x = r.standard_normal((M, D))
        y = r.standard_normal((N, D))
        b = r.standard_normal((N, E))
        a, S = orc.gauss_sum(x, y, b, sigma)
        Kd = np.exp(-cdist(x, y, "sqeuclidean") / sigma ** 2)
        _close(a, Kd @ b, 1e-12, 1e-14, "dense product")
        _close(S, Kd @ np.abs(b), 1e-12, 1e-14, "dense scale")


def pin_sum_bounds_unit_weights(orc):
    """b = 1: every kernel value lies in (0, 1], so 0 < a_i <= N, and a_i >= 1 when x_i is one of the y."""
    r = _rng(3)
    y = r.standard_normal((40, 3))
    x = np.concatenate([y[:5], r.standard_normal((10, 3))])
    a, _ = orc.gauss_sum(x, y, np.ones((40, 1)), 0.8)
    assert (a > 0).all() and (a <= 40).all()
    assert (a[:5] >= 1.0).all()


def pin_sum_translation_invariance(orc):
    r = _rng(4)
    x = r.standard_normal((6, 3))
    y = r.standard_normal((20, 3))
    b = r.standard_normal((20, 2))
    t = np.array([3.0, -7.5, 11.25])
    a0, _ = orc.gauss_sum(x, y, b, 1.3)
    a1, _ = orc.gauss_sum(x + t, y + t, b, 1.3)
    _close(a1, a0, 1e-12, 1e-14, "translation")


def pin_sum_scale_law(orc):
    """a(x, y; sigma) = a(x/sigma, y/sigma; 1)."""
    r = _rng(5)
    x = r.standard_normal((6, 4))
    y = r.standard_normal((25, 4))
    b = r.standard_normal((25, 1))
    s = 0.4
    a0, _ = orc.gauss_sum(x, y, b, s)
    a1, _ = orc.gauss_sum(x / s, y / s, b, 1.0)
    _close(a1, a0, 1e-12, 1e-14, "scale law")


def pin_sum_permutation_and_linearity(orc):
    """Permuting the (y_j, b_j) pairs changes nothing; a is linear in b."""
    r = _rng(6)
    x = r.standard_normal((5, 2))
    y = r.standard_normal((30, 2))
    b1 = r.standard_normal((30, 1))
    b2 = r.standard_normal((30, 1))
    p = r.permutation(30)
    a, _ = orc.gauss_sum(x, y, b1, 0.9)
    ap, _ = orc.gauss_sum(x, y[p], b1[p], 0.9)
    _close(ap, a, 1e-12, 1e-14, "permutation")
    a2, _ = orc.gauss_sum(x, y, b2, 0.9)
    al, _ = orc.gauss_sum(x, y, b1 - 2.5 * b2, 0.9)
    _close(al, a - 2.5 * a2, 1e-12, 1e-13, "linearity")


def pin_sum_columns_independent(orc):
    """An E-column call equals E one-column calls (the column index is not mixed with j)."""
    r = _rng(7)
    x = r.standard_normal((4, 3))
    y = r.standard_normal((9, 3))
    b = r.standard_normal((9, 3))
    a, S = orc.gauss_sum(x, y, b, 1.1)
    for e in range(3):
        ae, Se = orc.gauss_sum(x, y, b[:, e:e + 1], 1.1)
        assert np.array_equal(ae[:, 0], a[:, e]) and np.array_equal(Se[:, 0], S[:, e])


def pin_sum_scale_output(orc):
    """S = sum_j |k b| bounds |a| and equals a for non-negative b."""
    r = _rng(8)
    x = r.standard_normal((5, 3))
    y = r.standard_normal((30, 3))
    b = r.standard_normal((30, 1))
    a, S = orc.gauss_sum(x, y, b, 1.0)
    assert (S >= np.abs(a) - 1e-15).all()
    a2, S2 = orc.gauss_sum(x, y, np.abs(b), 1.0)
    _close(S2, a2, 1e-14, 0, "scale = a for b >= 0")
    _close(S, a2, 1e-14, 0, "scale = sum |k||b|")


def pin_sum_empty(orc):
    a, S = orc.gauss_sum(np.zeros((3, 2)), np.zeros((0, 2)), np.zeros((0, 1)), 1.0)
    assert (a == 0).all() and (S == 0).all()


# ---------------------------------------------------------------------------
# LogSumExp reduction
# ---------------------------------------------------------------------------
def pin_lse_golden(orc):
    for case in _golden()["lse"]:
        L = orc.gauss_lse(case["x"], case["y"], case["w"], case["sigma"])
        want = np.array([[_val(e) for e in row] for row in case["expect"]])
        _close(L, want, 1e-14, 1e-14, case["name"])


def pin_lse_is_log_of_sum(orc):
    """For b > 0: log sum_j k_ij b_j = LogSumExp with weight log b (ties LSE to the pinned Sum)."""
    r = _rng(9)
    x = r.standard_normal((8, 3))
    y = r.standard_normal((50, 3))
    b = 0.1 + 0.9 * r.random((50, 2))
    a, _ = orc.gauss_sum(x, y, b, 0.6)
    L = orc.gauss_lse(x, y, np.log(b), 0.6)
    _close(L, np.log(a), 1e-12, 1e-12, "lse = log sum")


def pin_lse_shift_and_stability(orc):
    """LSE(w + c) = LSE(w) + c, including shifts far outside exp's range."""
    r = _rng(10)
    x = r.standard_normal((5, 2))
    y = r.standard_normal((20, 2))
    w = r.standard_normal((20, 1))
    L0 = orc.gauss_lse(x, y, w, 0.7)
    for c in (3.5, 1000.0, -1000.0):
        L1 = orc.gauss_lse(x, y, w + c, 0.7)
        _close(L1, L0 + c, 1e-13, 1e-9, f"shift {c}")


def pin_lse_equal_terms(orc):
    """All N terms equal: LSE = t + log N."""
    y = np.tile(np.array([[1.0, -2.0, 0.5]]), (17, 1))
    x = np.array([[0.0, 0.0, 0.0]])
    L = orc.gauss_lse(x, y, np.full((17, 1), 0.25), 2.0)
    _close(L[0, 0], -(1 + 4 + 0.25) / 4.0 + 0.25 + math.log(17), 1e-14, 0, "equal terms")


def pin_lse_columns_and_empty(orc):
    r = _rng(11)
    x = r.standard_normal((3, 2))
    y = r.standard_normal((7, 2))
    w = r.standard_normal((7, 2))
    L = orc.gauss_lse(x, y, w, 1.0)
    for e in range(2):
        assert np.array_equal(orc.gauss_lse(x, y, w[:, e:e + 1], 1.0)[:, 0], L[:, e])
    L0 = orc.gauss_lse(x, np.zeros((0, 2)), np.zeros((0, 1)), 1.0)
    assert np.isneginf(L0).all()


# ---------------------------------------------------------------------------
# x-gradient
# ---------------------------------------------------------------------------
def pin_grad_golden(orc):
    for case in _golden()["grad_x"]:
        gx, G = orc.gauss_grad_x(case["x"], case["y"], case["b"], case["g"], case["sigma"])
        want = np.array([[_val(e) for e in row] for row in case["expect"]])
        _close(gx, want, 1e-14, 1e-15, case["name"])


def pin_grad_finite_differences(orc):
    """gx = d/dx of L(x) = sum_ie g_ie a_ie(x), by central differences of the pinned Sum."""
    r = _rng(12)
    M, N, D, E, sigma = 4, 30, 3, 2, 0.8
    x = r.standard_normal((M, D))
    y = r.standard_normal((N, D))
    b = r.standard_normal((N, E))
    g = r.standard_normal((M, E))
    gx, G = orc.gauss_grad_x(x, y, b, g, sigma)
    h = 1e-5
    fd = np.zeros_like(x)
    for i in range(M):
        for d in range(D):
            xp = x.copy(); xp[i, d] += h
            xm = x.copy(); xm[i, d] -= h
            ap, _ = orc.gauss_sum(xp, y, b, sigma)
            am, _ = orc.gauss_sum(xm, y, b, sigma)
            fd[i, d] = np.sum(g * (ap - am)) / (2 * h)
    assert (np.abs(gx - fd) <= 1e-7 * G + 1e-10).all(), np.max(np.abs(gx - fd))


def pin_grad_of_sum_of_squares(orc):
    """The README example: grad of sum_i a_i^2 is the gradient with g = 2a (checked by FD)."""
    r = _rng(13)
    x = r.standard_normal((3, 3))
    y = r.standard_normal((20, 3))
    b = np.ones((20, 1))
    a, _ = orc.gauss_sum(x, y, b, 1.0)
    gx, _ = orc.gauss_grad_x(x, y, b, 2 * a, 1.0)
    h = 1e-5
    for i in range(3):
        for d in range(3):
            xp = x.copy(); xp[i, d] += h
            xm = x.copy(); xm[i, d] -= h
            fd = (np.sum(orc.gauss_sum(xp, y, b, 1.0)[0] ** 2)
                  - np.sum(orc.gauss_sum(xm, y, b, 1.0)[0] ** 2)) / (2 * h)
            assert abs(gx[i, d] - fd) <= 1e-7 * max(1.0, abs(fd)), (i, d, gx[i, d], fd)


def pin_grad_stationary_and_translation(orc):
    """x_i = y_j with N = 1 is a stationary point; gradients are translation invariant."""
    r = _rng(14)
    y = r.standard_normal((1, 4))
    gx, _ = orc.gauss_grad_x(y.copy(), y, np.ones((1, 1)), np.ones((1, 1)), 0.5)
    assert (gx == 0).all()
    x = r.standard_normal((5, 3))
    y = r.standard_normal((12, 3))
    b = r.standard_normal((12, 1))
    g = r.standard_normal((5, 1))
    t = np.array([5.0, -3.0, 0.5])
    g0, G0 = orc.gauss_grad_x(x, y, b, g, 1.2)
    g1, _ = orc.gauss_grad_x(x + t, y + t, b, g, 1.2)
    assert (np.abs(g1 - g0) <= 1e-11 * G0 + 1e-14).all()
    assert (G0 >= np.abs(g0) - 1e-15).all()


# ---------------------------------------------------------------------------
# y-gradient and b-gradient (transposed product)
# ---------------------------------------------------------------------------
def pin_grad_y_golden(orc):
    for case in _golden()["grad_y"]:
        gy, G = orc.gauss_grad_y(case["x"], case["y"], case["b"], case["g"], case["sigma"])
        want = np.array([[_val(e) for e in row] for row in case["expect"]])
        _close(gy, want, 1e-14, 1e-15, case["name"])


def pin_grad_y_finite_differences(orc):
    """gy = d/dy of L(y) = sum_ie g_ie a_ie(y), by central differences of the pinned Sum."""
    r = _rng(18)
    M, N, D, E, sigma = 9, 5, 3, 2, 0.7
    x = r.standard_normal((M, D))
    y = r.standard_normal((N, D))
    b = r.standard_normal((N, E))
    g = r.standard_normal((M, E))
    gy, G = orc.gauss_grad_y(x, y, b, g, sigma)
    h = 1e-5
    fd = np.zeros_like(y)
    for j in range(N):
        for d in range(D):
            yp = y.copy(); yp[j, d] += h
            ym = y.copy(); ym[j, d] -= h
            ap, _ = orc.gauss_sum(x, yp, b, sigma)
            am, _ = orc.gauss_sum(x, ym, b, sigma)
            fd[j, d] = np.sum(g * (ap - am)) / (2 * h)
    assert (np.abs(gy - fd) <= 1e-7 * G + 1e-10).all(), np.max(np.abs(gy - fd))
    assert (G >= np.abs(gy) - 1e-15).all()


def pin_grad_xy_balance(orc):
    """Moving both clouds by the same vector leaves a unchanged, so the x- and
    y-gradients of any sum g.a add up to zero over the points, coordinate by coordinate."""
    r = _rng(19)
    x = r.standard_normal((11, 4))
    y = r.standard_normal((7, 4))
    b = r.standard_normal((7, 3))
    g = r.standard_normal((11, 3))
    gx, Gx = orc.gauss_grad_x(x, y, b, g, 1.1)
    gy, Gy = orc.gauss_grad_y(x, y, b, g, 1.1)
    tot = gx.sum(0) + gy.sum(0)
    assert (np.abs(tot) <= 1e-13 * (Gx.sum(0) + Gy.sum(0))).all(), tot


def pin_grad_y_rows_independent(orc):
    """Rows j of gy depend on row j of y and b only (a subset gives the same rows)."""
    r = _rng(20)
    x = r.standard_normal((6, 2))
    y = r.standard_normal((10, 2))
    b = r.standard_normal((10, 1))
    g = r.standard_normal((6, 1))
    gy, _ = orc.gauss_grad_y(x, y, b, g, 0.9)
    sub = [7, 2, 3]
    gs, _ = orc.gauss_grad_y(x, y[sub], b[sub], g, 0.9)
    assert np.array_equal(gs, gy[sub])


def pin_grad_b_golden(orc):
    for case in _golden()["grad_b"]:
        gb, S = orc.gauss_grad_b(case["x"], case["y"], case["g"], case["sigma"])
        want = np.array([[_val(e) for e in row] for row in case["expect"]])
        _close(gb, want, 1e-14, 1e-15, case["name"])


def pin_grad_b_linearity(orc):
    """a is linear in b, so L(b + t e_je) - L(b) = t gb_je exactly (up to rounding) for the
    pinned Sum; checked for every (j, e)."""
    r = _rng(21)
    M, N, D, E, sigma = 7, 6, 3, 2, 0.8
    x = r.standard_normal((M, D))
    y = r.standard_normal((N, D))
    b = r.standard_normal((N, E))
    g = r.standard_normal((M, E))
    gb, S = orc.gauss_grad_b(x, y, g, sigma)
    a0, _ = orc.gauss_sum(x, y, b, sigma)
    for j in range(N):
        for e in range(E):
            bp = b.copy(); bp[j, e] += 1.0
            a1, _ = orc.gauss_sum(x, y, bp, sigma)
            assert abs(np.sum(g * (a1 - a0)) - gb[j, e]) <= 1e-12 * (S[j, e] + 1), (j, e)


def pin_grad_b_bruteforce_scipy(orc):
    """Tiny inputs against SciPy's distance matrix: gb = K^T g."""
    from scipy.spatial.distance import cdist
    r = _rng(22)
    for (M, N, D, E, sigma) in [(8, 5, 3, 2, 0.6), (3, 12, 1, 1, 2.0)]:
        x = r.standard_normal((M, D))
        y = r.standard_normal((N, D))
        g = r.standard_normal((M, E))
        gb, S = orc.gauss_grad_b(x, y, g, sigma)
        Kd = np.exp(-cdist(x, y, "sqeuclidean") / sigma ** 2)
        _close(gb, Kd.T @ g, 1e-12, 1e-14, "transposed product")
        _close(S, Kd.T @ np.abs(g), 1e-12, 1e-14, "transposed scale")


# ---------------------------------------------------------------------------
# other radial kernels (Sum) and the Max / Min reductions
# ---------------------------------------------------------------------------
KERNEL_FNS = {   # written from each kernel's definition, for the brute-force pins
    "gaussian": lambda q, s: np.exp(-q / s ** 2),
    "laplace": lambda q, s: np.exp(-np.sqrt(q) / s),
    "cauchy": lambda q, s: 1.0 / (1.0 + q / s ** 2),
    "imq": lambda q, s: 1.0 / np.sqrt(1.0 + q / s ** 2),
}


def pin_kernel_sum_golden(orc):
    for case in _golden()["kernel_sum"]:
        for sigma, expect in zip(case["sigmas"], case["expect"]):
            a, _ = orc.kernel_sum(case["x"], case["y"], case["b"], sigma, case["kernel"])
            want = np.array([[_val(e) for e in row] for row in expect])
            _close(a, want, 1e-14, 0, f"{case['name']} sigma {sigma}")


def pin_kernel_sum_bruteforce_scipy(orc):
    """Every kernel against SciPy's distance matrix and a dense product."""
    from scipy.spatial.distance import cdist
    r = _rng(23)
    for kern, fn in KERNEL_FNS.items():
        for (M, N, D, E, sigma) in [(6, 13, 3, 2, 0.7), (9, 4, 5, 1, 2.0)]:
            x = r.standard_normal((M, D))
            y = r.standard_normal((N, D))
            b = r.standard_normal((N, E))
            a, S = orc.kernel_sum(x, y, b, sigma, kern)
            Kd = fn(cdist(x, y, "sqeuclidean"), sigma)
            _close(a, Kd @ b, 1e-12, 1e-14, f"{kern} dense product")
            _close(S, Kd @ np.abs(b), 1e-12, 1e-14, f"{kern} dense scale")


def pin_kernel_sum_gaussian_matches(orc):
    """kind 0 is the Gaussian of the pinned Sum."""
    r = _rng(24)
    x, y, b = r.standard_normal((5, 3)), r.standard_normal((17, 3)), r.standard_normal((17, 2))
    a0, S0 = orc.gauss_sum(x, y, b, 0.9)
    a1, S1 = orc.kernel_sum(x, y, b, 0.9, "gaussian")
    _close(a1, a0, 1e-15, 0, "gaussian kind")


def pin_laplace_lattice_sum(orc):
    """On a uniform 1-D lattice of spacing h through x, sum_k h exp(-|k| h / sigma)
    = h coth(h / (2 sigma)) (a geometric series); the lattice runs to 45 sigma, so the
    truncated tails are below 1e-19.  Fixes the square root and the sigma convention."""
    for sigma, h in ((0.8, 0.1), (2.0, 0.37)):
        n = int(45 * sigma / h)
        y = (h * np.arange(-n, n + 1))[:, None] + 0.25
        a, _ = orc.kernel_sum(np.array([[0.25]]), y, np.full((2 * n + 1, 1), h), sigma, "laplace")
        _close(a[0, 0], h / math.tanh(h / (2 * sigma)), 1e-12, 0, f"laplace lattice sigma {sigma}")


def pin_cauchy_lattice_sum(orc):
    """sum_{|k| <= n} h / (1 + (k h / sigma)^2) = h a^2 [ (pi / a) coth(pi a) - 2 Im psi(n + 1 + i a) / a ]
    with a = sigma / h: the Mittag-Leffler series of coth minus its tail, the tail
    written with the digamma function (SciPy, complex argument)."""
    from scipy.special import psi
    for sigma, h, n in ((0.5, 0.1, 400), (1.5, 0.25, 1000)):
        y = (h * np.arange(-n, n + 1))[:, None] - 1.0
        a, _ = orc.kernel_sum(np.array([[-1.0]]), y, np.full((2 * n + 1, 1), h), sigma, "cauchy")
        al = sigma / h
        full = (math.pi / al) / math.tanh(math.pi * al)
        tail = psi(complex(n + 1, al)).imag / al
        _close(a[0, 0], h * al * al * (full - 2 * tail), 1e-11, 0, f"cauchy lattice sigma {sigma}")


def pin_imq_squared_is_cauchy(orc):
    """One point: the inverse multiquadric squared is the Cauchy kernel; both are 1 at x = y
    and lie in (0, 1], so with b = 1 the sums lie in (0, N]."""
    r = _rng(25)
    x = r.standard_normal((7, 4))
    y = r.standard_normal((1, 4))
    ai, _ = orc.kernel_sum(x, y, np.ones((1, 1)), 1.3, "imq")
    ac, _ = orc.kernel_sum(x, y, np.ones((1, 1)), 1.3, "cauchy")
    _close(ai ** 2, ac, 1e-14, 0, "imq^2 = cauchy")
    yy = r.standard_normal((30, 4))
    for kern in KERNEL_FNS:
        a, _ = orc.kernel_sum(yy[:3], yy, np.ones((30, 1)), 0.6, kern)
        assert (a >= 1.0).all() and (a <= 30).all(), kern
        a1, _ = orc.kernel_sum(yy[:1], yy[:1], np.full((1, 1), 2.5), 0.6, kern)
        assert a1[0, 0] == 2.5, kern


def pin_kernel_sum_scale_law(orc):
    """a(x, y; sigma) = a(x / sigma, y / sigma; 1) for every kernel (all are functions of |x - y| / sigma)."""
    r = _rng(26)
    x, y, b = r.standard_normal((4, 3)), r.standard_normal((21, 3)), r.standard_normal((21, 1))
    for kern in KERNEL_FNS:
        a0, _ = orc.kernel_sum(x, y, b, 0.45, kern)
        a1, _ = orc.kernel_sum(x / 0.45, y / 0.45, b, 1.0, kern)
        _close(a1, a0, 1e-12, 1e-14, f"{kern} scale law")


def pin_maxmin_golden(orc):
    for case in _golden()["maxmin"]:
        for red in ("max", "min"):
            val, idx, second = orc.kernel_maxmin(case["x"], case["y"], case["b"], case["sigma"], case["kernel"], red)
            want = case[red]
            _close(val[:, 0], [_val(v) for v in want["val"]], 1e-15, 0, f"{case['name']} {red}")
            assert idx[:, 0].tolist() == want["idx"], (case["name"], red, idx)
            _close(second[:, 0], [_val(v) for v in want["second"]], 1e-15, 0, f"{case['name']} {red} second")


def pin_maxmin_bruteforce_numpy(orc):
    """Against NumPy's max/argmax (first occurrence) on the dense formula, including
    exact ties from points on an integer grid."""
    from scipy.spatial.distance import cdist
    r = _rng(27)
    for kern, fn in KERNEL_FNS.items():
        x = r.integers(-2, 3, size=(12, 2)).astype(float)
        y = r.integers(-2, 3, size=(40, 2)).astype(float)
        b = r.integers(-2, 3, size=(40, 3)).astype(float)
        F = fn(cdist(x, y, "sqeuclidean"), 1.1)[:, :, None] * b[None, :, :]
        for red, pick, arg in (("max", np.max, np.argmax), ("min", np.min, np.argmin)):
            val, idx, second = orc.kernel_maxmin(x, y, b, 1.1, kern, red)
            _close(val, pick(F, axis=1), 1e-14, 1e-300, f"{kern} {red}")
            assert np.array_equal(idx, arg(F, axis=1)), (kern, red)
            for i in range(12):
                for e in range(3):
                    rest = np.delete(F[i, :, e], idx[i, e])
                    _close(second[i, e], pick(rest), 1e-14, 1e-300, f"{kern} {red} runner-up")


def pin_max_unit_weights_is_nearest(orc):
    """b = 1: every kernel decreases with distance, so ArgMax is the nearest point (the
    pinned K-min with K = 1, same lowest-index rule) and the Max is k at that distance."""
    r = _rng(28)
    x = np.round(r.standard_normal((15, 3)) * 2) / 2
    y = np.round(r.standard_normal((50, 3)) * 2) / 2
    i1, d1, _ = orc.knn(x, y, 1)
    for kern, fn in KERNEL_FNS.items():
        val, idx, _ = orc.kernel_maxmin(x, y, np.ones((50, 1)), 0.8, kern, "max")
        assert np.array_equal(idx[:, 0], i1[:, 0]), kern
        _close(val[:, 0], fn(d1[:, 0], 0.8), 1e-14, 0, kern)


def pin_min_is_negated_max(orc):
    """Min(k b) = -Max(k (-b)) with the same index; N = 0 gives -inf / +inf and -1."""
    r = _rng(29)
    x, y, b = r.standard_normal((6, 3)), r.standard_normal((25, 3)), r.standard_normal((25, 2))
    vmin, imin, smin = orc.kernel_maxmin(x, y, b, 0.7, "cauchy", "min")
    vmax, imax, smax = orc.kernel_maxmin(x, y, -b, 0.7, "cauchy", "max")
    assert np.array_equal(vmin, -vmax) and np.array_equal(imin, imax) and np.array_equal(smin, -smax)
    v, i, _ = orc.kernel_maxmin(x, np.zeros((0, 3)), np.zeros((0, 2)), 1.0, "gaussian", "max")
    assert np.isneginf(v).all() and (i == -1).all()
    v, i, _ = orc.kernel_maxmin(x, np.zeros((0, 3)), np.zeros((0, 2)), 1.0, "gaussian", "min")
    assert np.isposinf(v).all() and (i == -1).all()


# ---------------------------------------------------------------------------
# block-sparse (cluster ranges) Sum / Max / Min
# ---------------------------------------------------------------------------
def _random_ranges(r, M, N, nc, max_ranges, overlap=True):
    """Row clusters covering a random subset of [0, M) and random column ranges."""
    cuts = np.sort(r.choice(np.arange(1, M), size=2 * nc - 1, replace=False))
    edges = np.concatenate([[0], cuts, [M]])
    ranges_i = np.stack([edges[0:-1:2], edges[1::2]], 1)[:nc]   # every other segment is a cluster
    slices, red = [], []
    for _ in range(nc):
        for _ in range(r.integers(0, max_ranges + 1)):
            a = int(r.integers(0, N))
            c = int(r.integers(a, N + 1)) if overlap else min(N, a + int(r.integers(0, 6)))
            red.append([a, c])
        slices.append(len(red))
    return ranges_i, np.array(slices), np.array(red, dtype=np.int64).reshape(-1, 2)


def _mask(M, N, ranges_i, slices_i, redranges_j):
    W = np.zeros((M, N))
    for c, (i0, i1) in enumerate(ranges_i):
        for rr in range(slices_i[c - 1] if c else 0, slices_i[c]):
            W[i0:i1, redranges_j[rr][0]:redranges_j[rr][1]] += 1
    covered = np.zeros(M, bool)
    for (i0, i1) in ranges_i:
        covered[i0:i1] = True
    return W, covered


def pin_ranges_golden(orc):
    for case in _golden()["ranges"]:
        args = (case["ranges_i"], case["slices_i"], case["redranges_j"])
        a, _ = orc.kernel_ranges(case["x"], case["y"], case["b"], case["sigma"], case["kernel"], "sum", *args)
        _close(a[:, 0], [_val(v) for v in case["sum"]], 1e-15, 0, case["name"])
        for red in ("max", "min"):
            v, i, _ = orc.kernel_ranges(case["x"], case["y"], case["b"], case["sigma"], case["kernel"], red, *args)
            _close(v[:2, 0], [_val(t) for t in case[red]["val"]], 1e-15, 0, f"{case['name']} {red}")
            assert i[:2, 0].tolist() == case[red]["idx"], (red, i)
            assert i[2, 0] == -1 and np.isinf(v[2, 0]) and (v[2, 0] > 0) == (red == "min")


def pin_ranges_mask_bruteforce(orc):
    """Against a dense masked product: W_ij = how many ranges of i's cluster contain j;
    a = (K o W) b, and Max / Min over the j with W_ij > 0 (NumPy, first occurrence)."""
    from scipy.spatial.distance import cdist
    r = _rng(30)
    for kern, fn in KERNEL_FNS.items():
        M, N = 40, 60
        x = np.round(r.standard_normal((M, 2)) * 2) / 2
        y = np.round(r.standard_normal((N, 2)) * 2) / 2
        b = np.round(r.standard_normal((N, 2)) * 2) / 2
        ri, si, rj = _random_ranges(r, M, N, 5, 3)
        W, covered = _mask(M, N, ri, si, rj)
        Kd = fn(cdist(x, y, "sqeuclidean"), 0.9)
        a, S = orc.kernel_ranges(x, y, b, 0.9, kern, "sum", ri, si, rj)
        _close(a, (Kd * W) @ b, 1e-12, 1e-14, f"{kern} masked sum")
        _close(S, (Kd * W) @ np.abs(b), 1e-12, 1e-14, f"{kern} masked scale")
        for red, big in (("max", -np.inf), ("min", np.inf)):
            v, i, _ = orc.kernel_ranges(x, y, b, 0.9, kern, red, ri, si, rj)
            for e in range(2):
                F = np.where(W > 0, Kd * b[:, e][None, :], big)
                pick = (np.argmax if red == "max" else np.argmin)(F, axis=1)
                has = (W > 0).any(1)
                assert np.array_equal(i[:, e], np.where(has, pick, -1)), (kern, red)
                want = np.where(has, F[np.arange(M), pick], big)
                _close(v[:, e], want, 1e-14, 1e-300, f"{kern} {red} masked")


def pin_ranges_split_invariance(orc):
    """Cutting a column range in two, or a row cluster in two with the same ranges, leaves
    the Sum (to rounding) and the Max and its index (exactly) unchanged; one cluster over
    all rows with one range over all columns is the dense reduction."""
    r = _rng(31)
    x, y, b = r.standard_normal((20, 3)), r.standard_normal((50, 3)), r.standard_normal((50, 1))
    base = ([[0, 20]], [2], [[5, 40], [30, 50]])
    cut_j = ([[0, 20]], [3], [[5, 17], [17, 40], [30, 50]])
    cut_i = ([[0, 8], [8, 20]], [2, 4], [[5, 40], [30, 50], [5, 40], [30, 50]])
    a0, _ = orc.kernel_ranges(x, y, b, 1.2, "laplace", "sum", *base)
    v0, i0, _ = orc.kernel_ranges(x, y, b, 1.2, "laplace", "max", *base)
    for alt in (cut_j, cut_i):
        a1, _ = orc.kernel_ranges(x, y, b, 1.2, "laplace", "sum", *alt)
        _close(a1, a0, 1e-13, 1e-15, "split invariance")
        v1, i1, _ = orc.kernel_ranges(x, y, b, 1.2, "laplace", "max", *alt)
        assert np.array_equal(v1, v0) and np.array_equal(i1, i0)
    a, _ = orc.kernel_ranges(x, y, b, 1.2, "gaussian", "sum", [[0, 20]], [1], [[0, 50]])
    _close(a, orc.gauss_sum(x, y, b, 1.2)[0], 1e-15, 0, "dense cover")


# ---------------------------------------------------------------------------
# K-min / ArgMin
# ---------------------------------------------------------------------------
def pin_knn_golden(orc):
    for case in _golden()["knn"]:
        idx, dist, nxt = orc.knn(case["x"], case["y"], case["K"])
        assert idx.tolist() == case["expect_idx"], (case["name"], idx)
        _close(dist, [[_val(v) for v in row] for row in case["expect_dist"]], 0, 0, case["name"])
        _close(nxt, [_val(v) for v in case["expect_next"]], 0, 0, case["name"] + " next")


def pin_knn_full_sort(orc):
    """K = N: the result is the stable argsort of the row's distances (NumPy)."""
    r = _rng(15)
    x = np.round(r.standard_normal((6, 3)) * 4) / 4      # coarse grid: many exact ties
    y = np.round(r.standard_normal((40, 3)) * 4) / 4
    idx, dist, nxt = orc.knn(x, y, 40)
    for i in range(6):
        d = ((x[i] - y) ** 2).sum(1)
        order = np.argsort(d, kind="stable")
        assert idx[i].tolist() == order.tolist()
        assert np.array_equal(dist[i], d[order])
        assert np.isinf(nxt[i])


def pin_knn_kdtree(orc):
    """Against SciPy's k-d tree (a different algorithm) on tie-free random data."""
    from scipy.spatial import cKDTree
    r = _rng(16)
    x = r.standard_normal((20, 4))
    y = r.standard_normal((300, 4))
    idx, dist, nxt = orc.knn(x, y, 7)
    dd, ii = cKDTree(y).query(x, k=8)
    assert np.array_equal(idx, ii[:, :7])
    _close(np.sqrt(dist), dd[:, :7], 1e-12, 1e-12, "kd distances")
    _close(np.sqrt(nxt), dd[:, 7], 1e-12, 1e-12, "kd next")


def pin_knn_ties_and_self(orc):
    """Duplicated points come out lowest index first; x_i = y_j gives (j, 0) first."""
    y = np.array([[1.0, 1.0], [5.0, 5.0], [1.0, 1.0], [0.0, 0.0], [1.0, 1.0], [9.0, 9.0]])
    idx, dist, nxt = orc.knn(np.array([[1.0, 1.0], [5.0, 5.0]]), y, 3)
    assert idx.tolist() == [[0, 2, 4], [1, 0, 2]], idx
    assert dist[0].tolist() == [0.0, 0.0, 0.0] and nxt[0] == 2.0
    idx1, _, _ = orc.knn(np.array([[0.9, 0.9]]), y, 1)        # ArgMin = K-min with K = 1
    assert idx1.tolist() == [[0]]


def pin_knn_translation(orc):
    """Integer coordinates keep distances exact, so a shift leaves the indices unchanged."""
    r = _rng(17)
    x = r.integers(-5, 6, size=(8, 3)).astype(float)
    y = r.integers(-5, 6, size=(60, 3)).astype(float)
    i0, d0, n0 = orc.knn(x, y, 5)
    i1, d1, n1 = orc.knn(x + 100, y + 100, 5)
    assert np.array_equal(i0, i1) and np.array_equal(d0, d1) and np.array_equal(n0, n1)


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]

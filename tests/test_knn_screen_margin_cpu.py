"""The tensor-core K-min screen's error bound, checked on the host (no GPU).

The screen forms S_ij = A_i . B_j from the high fp16 halves of the augmented operands
A_i = [2 x_i, -|x_i|^2, -1] and B_j = [y_j, 1, |y_j|^2] (|.|^2 summed in fp32, then rounded to
fp16 like every other entry), accumulated in fp32, and passes point j when -S_ij is at most the
row's current K-th direct distance plus
    margin_i = 2^-8 (|x_i|^2 + max_j |y_j|^2) + 2^-24 (D + 2).
No point of the row's final K may fail, so for every pair -S_ij must stay within margin_i of the
direct fp32 distance q_ij = sum over d of (x_id - y_jd)^2 (summed in coordinate order): the
margin has to cover the fp16 rounding of the operands and the fp32 accumulation.  Here the
products of fp16 values are formed exactly (fp64), their sum is bounded by the worst fp32
accumulation of 64 terms (each step within 2^-23 of the running magnitude: round to nearest or
toward zero), and q_ij is formed in fp32 as the kernel forms it; the check is
|sum + q_ij| + accumulation bound <= margin_i over clouds of many scales: unit, subnormal in
fp16, near the norm limit of 4096, spread log-uniformly over seven decades, and coordinates
placed half a unit in the last place of fp16 away from representable values.
"""
import numpy as np
import pytest

NORM_LIMIT = 4096.0


def _fp32_sq_norm(v):
    """sum of c^2 in fp32, one rounding a step (an fma: the product is exact in fp64)"""
    n = np.float32(0.0)
    for c in v.astype(np.float32):
        n = np.float32(np.float64(c) * np.float64(c) + np.float64(n))
    return n


def _fp32_direct(xi, yj):
    q = np.float32(0.0)
    for a, b in zip(xi.astype(np.float32), yj.astype(np.float32)):
        df = np.float32(a - b)
        q = np.float32(np.float64(df) * np.float64(df) + np.float64(q))  # one rounding: an fma
    return q


def _operands(x, y):
    """High fp16 halves of A (rows of x) and B (rows of y), as fp64 arrays of K = 64."""
    M, D = x.shape
    N = y.shape[0]
    nx = np.array([_fp32_sq_norm(r) for r in x], dtype=np.float32)
    ny = np.array([_fp32_sq_norm(r) for r in y], dtype=np.float32)
    A = np.zeros((M, 64), dtype=np.float32)
    B = np.zeros((N, 64), dtype=np.float32)
    A[:, :D] = np.float32(2.0) * x
    A[:, D] = -nx
    A[:, D + 1] = -1.0
    B[:, :D] = y
    B[:, D] = 1.0
    B[:, D + 1] = ny
    return A.astype(np.float16).astype(np.float64), B.astype(np.float16).astype(np.float64), nx, ny


def _worst_ratio(x, y):
    """max over pairs of (|-S_exact - q| + accumulation bound) / margin."""
    M, D = x.shape
    Ah, Bh, nx, ny = _operands(x, y)
    margin = 2.0 ** -8 * (nx.astype(np.float64) + float(ny.max())) + 2.0 ** -24 * (D + 2)
    worst = 0.0
    for i in range(M):
        terms = Ah[i][None, :] * Bh  # exact products of fp16 values
        s = terms.sum(1)
        acc = 63 * 2.0 ** -23 * np.abs(terms).sum(1)
        q = np.array([_fp32_direct(x[i], y[j]) for j in range(y.shape[0])], dtype=np.float64)
        err = np.abs(-s - q) + acc
        worst = max(worst, float(np.max(err / margin[i])))
    return worst


def _clouds(kind, rng, M=12, N=40, D=50):
    if kind == "unit":
        x, y = rng.standard_normal((M, D)) / np.sqrt(D), rng.standard_normal((N, D)) / np.sqrt(D)
    elif kind == "subnormal":  # every fp16 operand below 2^-14
        x, y = 1e-5 * rng.standard_normal((M, D)), 1e-5 * rng.standard_normal((N, D))
    elif kind == "near_limit":  # max |x|^2 + max |y|^2 just under 4096
        x, y = rng.standard_normal((M, D)), rng.standard_normal((N, D))
        s = np.sqrt(0.49 * NORM_LIMIT / max((x ** 2).sum(1).max(), (y ** 2).sum(1).max()))
        x, y = s * x, s * y
    elif kind == "log_uniform":
        def f(n):
            return np.sign(rng.standard_normal((n, D))) * 10.0 ** rng.uniform(-7, 0, (n, D))
        x, y = f(M), f(N)
    elif kind == "half_ulp":  # 1 + (k + 1/2) 2^-10: halfway between fp16 neighbours
        def f(n):
            k = rng.integers(0, 1023, size=(n, D))
            return np.sign(rng.standard_normal((n, D))) * (1.0 + (k + 0.5) * 2.0 ** -10) / np.sqrt(D)
        x, y = f(M), f(N)
    elif kind == "close_pairs":  # near neighbours: q far below the norms
        base = rng.standard_normal((N, D))
        y = base
        x = base[rng.integers(0, N, size=M)] + 1e-3 * rng.standard_normal((M, D))
    else:
        raise ValueError(kind)
    return x.astype(np.float32), y.astype(np.float32)


@pytest.mark.parametrize("kind", ["unit", "subnormal", "near_limit", "log_uniform", "half_ulp", "close_pairs"])
def test_screen_error_within_margin(kind):
    seeds = {"unit": 1, "subnormal": 2, "near_limit": 3, "log_uniform": 4, "half_ulp": 5, "close_pairs": 6}
    rng = np.random.default_rng(seeds[kind])
    x, y = _clouds(kind, rng)
    if kind == "near_limit":
        nx = (x.astype(np.float64) ** 2).sum(1).max()
        ny = (y.astype(np.float64) ** 2).sum(1).max()
        assert 0.9 * NORM_LIMIT <= nx + ny <= NORM_LIMIT
    assert _worst_ratio(x, y) <= 1.0


def test_margin_is_not_loose_by_orders_of_magnitude():
    """The relative part is needed: a margin 64 times smaller fails on clouds whose operands
    sit halfway between fp16 neighbours."""
    rng = np.random.default_rng(3)
    x, y = _clouds("half_ulp", rng)
    assert _worst_ratio(x, y) * 64 > 1.0

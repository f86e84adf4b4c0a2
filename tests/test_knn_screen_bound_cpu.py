"""The K-min screen's bound, on CPU, by emulating the kernel's fp32 arithmetic.

The filtered K-min skips a group of points when every point's filter value
f = h_j + sum_d x~_d (-y~_d)  (h_j = fl(|y~_j|^2) (1 - kappa) / 2)  exceeds
T = ((thr + 2^-100 + kappa (|x~|^2 + thr)) - |x~|^2) / 2, thr being the row's current K-th
direct fp32 distance.  This is safe only if f > T implies that the point's direct fp32
distance is >= thr (it could not have been inserted).  Here the kernel's operations are
replayed in fp32 (an FMA as the exact product plus one rounding) on millions of pairs from
adversarial clouds (a common offset, norms over twelve decades, ulp-spaced shells around the
threshold), with thr placed at and next to the pairs' own distances, and the implication is
checked for every pair.  The constants are the kernel's: kappa = (8 D + 12) 2^-24."""
import numpy as np
import pytest

U = 2.0 ** -24


def _fma(a, b, c):
    """fp32 fused multiply-add: the product is exact in fp64, then one rounding (fp64 add
    first; a second rounding differs from the true FMA in fewer than 1 in 2^28 cases)."""
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def _chains(DP):
    return 4 if DP >= 32 else 2 if DP >= 16 else 1


def _dot_chain(prod_pairs, start, DP):
    """sum of prod terms in the kernel's interleaved chains: chain 0 starts at `start`
    (fma), chains c > 0 start with a rounded product; then the chains are added in order."""
    nc = _chains(DP)
    acc = [None] * nc
    for d, (a, b) in enumerate(prod_pairs):
        c = d % nc
        if d < nc:
            acc[c] = _fma(a, b, start) if c == 0 else (a.astype(np.float32) * b).astype(np.float32)
        else:
            acc[c] = _fma(a, b, acc[c])
    s = acc[0]
    for c in range(1, nc):
        s = (s + acc[c]).astype(np.float32)
    return s


def _sq_norm(v):
    """fl(|v|^2) as the kernel's fma chain (first product rounded)."""
    s = (v[..., 0] * v[..., 0]).astype(np.float32)
    for d in range(1, v.shape[-1]):
        s = _fma(v[..., d], v[..., d], s)
    return s


def _direct(x, y, DP):
    """The direct fp32 distance of the kernels: fl(x - y) squared in interleaved chains."""
    df = (x[:, None, :] - y[None, :, :]).astype(np.float32)
    nc = _chains(DP)
    acc = [None] * nc
    for d in range(x.shape[1]):
        c = d % nc
        sq = df[..., d]
        acc[c] = (sq * sq).astype(np.float32) if d < nc else _fma(sq, sq, acc[c])
    s = acc[0]
    for c in range(1, nc):
        s = (s + acc[c]).astype(np.float32)
    return s


def _screen(x, y, thr):
    """f (rows x points) and T (rows) as the kernel computes them."""
    D = x.shape[1]
    DP = D if D <= 4 else 8 if D <= 8 else 16
    kappa = np.float32((8 * DP + 12) * U)
    kh = np.float32(0.5) * (np.float32(1.0) - kappa)
    c = x.mean(axis=0).astype(np.float32)                  # any centre is allowed by the bound
    xt = (x - c).astype(np.float32)
    yt = (y - c).astype(np.float32)
    yy = _sq_norm(yt)
    h = np.where(yy < np.float32(2.0 ** 100), (kh * yy).astype(np.float32), np.float32(-np.inf))
    pairs = [(np.broadcast_to(xt[:, None, d], (x.shape[0], y.shape[0])), np.broadcast_to(-yt[None, :, d],
              (x.shape[0], y.shape[0]))) for d in range(D)]
    f = _dot_chain(pairs, np.broadcast_to(h[None, :], (x.shape[0], y.shape[0])), DP)
    xx = _sq_norm(xt)
    s1 = (xx + thr).astype(np.float32)
    s2 = _fma(np.full_like(xx, kappa), s1, (thr + np.float32(2.0 ** -100)).astype(np.float32))
    T = (np.float32(0.5) * (s2 - xx).astype(np.float32)).astype(np.float32)
    T = np.where(xx < np.float32(2.0 ** 100), T, np.float32(np.inf))
    return f, T, DP


def _check(x, y, rng):
    x = x.astype(np.float32)
    y = y.astype(np.float32)
    D = x.shape[1]
    DP = D if D <= 4 else 8 if D <= 8 else 16
    d = _direct(x, y, DP)
    # thresholds at a pair's own distance and one ulp either side
    base = d[np.arange(x.shape[0]), rng.integers(0, y.shape[0], x.shape[0])]
    for thr in (base, np.nextafter(base, np.float32(np.inf)), np.nextafter(base, np.float32(0))):
        thr = thr.astype(np.float32)
        f, T, _ = _screen(x, y, thr)
        skipped = f > T[:, None]
        bad = skipped & (d < thr[:, None])
        assert not bad.any(), (f"screen skipped {int(bad.sum())} pairs that the direct test inserts "
                               f"(D={D}); first at {np.argwhere(bad)[0].tolist()}")


@pytest.mark.parametrize("D", [1, 2, 3, 4, 8, 16])
def test_normal_clouds(D):
    r = np.random.Generator(np.random.PCG64(10 + D))
    _check(r.standard_normal((128, D)), r.standard_normal((3000, D)), r)


@pytest.mark.parametrize("D", [2, 3, 16])
def test_common_offset(D):
    r = np.random.Generator(np.random.PCG64(20 + D))
    _check(1e3 + 1e-2 * r.standard_normal((128, D)), 1e3 + 1e-2 * r.standard_normal((3000, D)), r)


@pytest.mark.parametrize("D", [3, 8])
def test_norms_over_decades(D):
    r = np.random.Generator(np.random.PCG64(30 + D))

    def cloud(n):
        v = r.standard_normal((n, D))
        return v / np.linalg.norm(v, axis=1, keepdims=True) * 10.0 ** r.uniform(-6, 6, size=(n, 1))

    _check(cloud(128), cloud(3000), r)


@pytest.mark.parametrize("D", [2, 3, 4])
def test_ulp_shell_around_the_threshold(D):
    """Points on a shell of squared radii 1 + k 2^-23 around rows near the origin: thr lands
    among distances one ulp apart."""
    r = np.random.Generator(np.random.PCG64(40 + D))
    u = r.standard_normal((3000, D))
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    y = u * np.sqrt(1.0 + np.arange(3000) * 2.0 ** -23)[:, None]
    x = 1e-3 * r.standard_normal((128, D))
    _check(x, y, r)

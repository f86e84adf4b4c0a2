"""K-min at D <= 16 screens point groups with |y~|^2 - 2 x~.y~ (centred coordinates)
and inserts by the direct fp32 distance.  These cases aim at the screen's bound: a
common offset far larger than the distances, clouds whose norms span twelve decades,
points whose |y~|^2 or |x~|^2 is too large to bound (they must always pass), and
shells of distinct fp32 distances one ulp apart around the K-th.  Every case is
checked against the fp64 oracle with the K-min gate (exact indices wherever the
oracle's distances are separated)."""
import math
from fractions import Fraction

import numpy as np
import pytest

import symbolic_matrix_reductions_gb300 as kr

from parity import check_knn

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from symbolic_matrix_reductions_gb300 import build
    build.build()
    kr.load_library()


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _f32(q: Fraction) -> float:
    """q rounded to the nearest fp32 (ties to even), subnormals included."""
    if q == 0:
        return 0.0
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    if Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    m = a * Fraction(2) ** (23 - e)
    n, rem = divmod(m.numerator, m.denominator)
    if 2 * rem > m.denominator or (2 * rem == m.denominator and n % 2 == 1):
        n += 1
    v = math.ldexp(float(n), e - 23)
    return -v if q < 0 else v


def _direct_fp32(xr, yr, DP):
    """The kernels' direct distance in exact fp32 steps: fl(x_d - y_d), squared and
    summed in dist_chains(DP) interleaved fma chains, the chains added in order."""
    nc = 4 if DP >= 32 else 2 if DP >= 16 else 1
    qc = [None] * nc
    for d in range(DP):
        df = Fraction(_f32(Fraction(float(xr[d])) - Fraction(float(yr[d])))) if d < len(xr) else Fraction(0)
        c = d % nc
        qc[c] = _f32(df * df) if d < nc else _f32(df * df + Fraction(qc[c]))
    q = qc[0]
    for c in range(1, nc):
        q = _f32(Fraction(q) + Fraction(qc[c]))
    return q


def _pad(D):
    return D if D <= 4 else 8 if D <= 8 else 16


def _exact_list(x, y, K, rows):
    """For each row: the K smallest (direct fp32 distance, index) pairs, taken over
    the points within 1e-4 (relative) of the fp64 K-th distance."""
    DP = _pad(x.shape[1])
    out = {}
    for i in rows:
        d64 = ((x[i].astype(np.float64) - y.astype(np.float64)) ** 2).sum(axis=1)
        kth = np.partition(d64, K - 1)[K - 1]
        cand = np.nonzero(d64 <= kth * (1 + 1e-4) + 1e-300)[0]
        q = sorted((_direct_fp32(x[i], y[j], DP), int(j)) for j in cand)[:K]
        out[i] = q
    return out


def _run(orc, x, y, K, split, what, exact_rows=0):
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.ascontiguousarray(y, dtype=np.float32)
    xt, yt = (torch.from_numpy(a).to(DEV) for a in (x, y))
    idx, dist = kr.kernel_knn(xt, yt, K, split=split)
    torch.cuda.synchronize()
    idx, dist = idx.cpu().numpy(), dist.cpu().numpy()
    i_ref, d_ref, n_ref = orc.knn(x, y, K)
    ties = check_knn(idx, dist, x, y, i_ref, d_ref, n_ref, what)
    if exact_rows:
        # the list the unfiltered scan yields, bit for bit
        rows = np.random.Generator(np.random.PCG64(x.shape[0])).choice(x.shape[0], min(exact_rows, x.shape[0]),
                                                                       replace=False)
        for i, q in _exact_list(x, y, K, rows).items():
            assert [j for _, j in q] == idx[i].tolist(), f"{what}: row {i} indices {idx[i].tolist()} vs {q}"
            assert [v for v, _ in q] == dist[i].astype(np.float64).tolist(), f"{what}: row {i} distances"
    return ties


@pytest.mark.parametrize("D", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("split", [0, 3])
def test_common_offset(orc, D, split):
    """Offset 1e3, spread 1e-2: without the centring the bound would pass every group."""
    r = _rng(100 + D)
    x = 1e3 + 1e-2 * r.standard_normal((600, D))
    y = 1e3 + 1e-2 * r.standard_normal((3000, D))
    _run(orc, x, y, 10, split, f"offset D{D} S{split}", exact_rows=40)


@pytest.mark.parametrize("D,K", [(2, 10), (3, 1), (3, 10), (3, 32), (8, 16), (16, 10)])
def test_norms_over_twelve_decades(orc, D, K):
    r = _rng(200 + D + K)

    def cloud(n):
        v = r.standard_normal((n, D))
        v /= np.linalg.norm(v, axis=1, keepdims=True)
        return v * 10.0 ** r.uniform(-6, 6, size=(n, 1))

    _run(orc, cloud(500), cloud(2500), K, 0, f"decades D{D} K{K}", exact_rows=60)


@pytest.mark.parametrize("D", [3, 16])
def test_unboundable_points_always_pass(orc, D):
    """y rows with |y|^2 >= 2^100 (h = -inf) or overflowing to inf must never hide a
    nearer point, and are themselves never among the K nearest here; rows of x with
    |x|^2 >= 2^100 switch the screen off (T = +inf) for their whole block."""
    r = _rng(300 + D)
    x = r.standard_normal((700, D))
    y = r.standard_normal((4000, D))
    y[5] = 1e30            # |y|^2 overflows fp32
    y[777] = -1e18         # |y|^2 = D 1e36: finite, above 2^100
    y[3999, 0] = 3e15      # above 2^100 in one coordinate
    x[600] = 1e18          # a row of x above 2^100 (its block's screen is off)
    _run(orc, x, y, 10, 0, f"unboundable D{D}")


@pytest.mark.parametrize("D", [2, 3, 4])
def test_shell_of_ulp_spaced_distances(orc, D):
    """Rows at the origin and points at squared radius 1 + k 2^-23 (distinct fp32
    distances one ulp apart), shuffled: the screen's margin is a few ulps, so the
    K-th and its neighbours are decided by the direct distance alone."""
    r = _rng(400 + D)
    n = 3000
    u = r.standard_normal((n, D))
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    rad = np.sqrt(1.0 + np.arange(n) * 2.0 ** -23)
    y = (u * rad[:, None])[r.permutation(n)]
    x = np.zeros((130, D))
    x[1::2] = 1e-3 * r.standard_normal((65, D))
    _run(orc, x, y, 10, 0, f"shell D{D}", exact_rows=130)


def test_far_subset_and_duplicates(orc):
    """A tenth of y shifted by 1e4 (large |y~|^2 beside small ones in one tile) and
    every point of y duplicated once (equal distances: the lower index first)."""
    r = _rng(500)
    y = r.standard_normal((2000, 3))
    y[r.random(2000) < 0.1] += 1e4
    y = np.concatenate([y, y])
    x = r.standard_normal((900, 3))
    for split in (0, 4):
        _run(orc, x, y, 10, split, f"far+dup S{split}", exact_rows=60)


@pytest.mark.parametrize("D,split", [(3, 4), (16, 3), (8, 7)])
def test_split_with_all_neighbours_in_one_split(orc, D, split):
    """Split-j where every row's nearest points are in the first split's columns and the later
    splits hold only far points (their lists fill with far candidates): the merged lists must
    give the oracle's result."""
    r = np.random.Generator(np.random.PCG64(404 + D + split))
    M, N, K = 700, 9000, 10
    x = r.standard_normal((M, D)).astype(np.float32)
    near = (x[r.integers(0, M, size=2000)] + 0.01 * r.standard_normal((2000, D))).astype(np.float32)
    far = (5.0 + r.standard_normal((N - 2000, D))).astype(np.float32)
    y = np.concatenate([near, far])
    idx, dist = kr.kernel_knn(*(torch.from_numpy(a).to(DEV) for a in (x, y)), K, split=split)
    torch.cuda.synchronize()
    i_ref, d_ref, n_ref = orc.knn(x, y, K)
    check_knn(idx.cpu().numpy(), dist.cpu().numpy(), x, y, i_ref, d_ref, n_ref, f"one split near D{D} S{split}")

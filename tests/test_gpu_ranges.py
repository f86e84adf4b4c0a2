"""Block-sparse (cluster ranges) Sum / Max / Min vs the fp64 oracle, through the C ABI:
random clusters with overlapping and out-of-order column ranges, rows in no cluster,
empty clusters, clusters longer than a thread block, and a truncated kernel product
on spatially sorted points (the use the pages describe)."""
import numpy as np
import pytest

import symbolic_matrix_reductions_gb300 as kr

from parity import check_maxmin, check_sum

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"
KINDS = ["gaussian", "laplace", "cauchy", "imq"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from symbolic_matrix_reductions_gb300 import build
    build.build()
    kr.load_library()


@pytest.fixture(scope="module")
def orc():
    import oracle
    return oracle.load()


def _np(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def _t(*arrs):
    return [torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in arrs]


def _tables(r, M, N, nc, max_ranges):
    """nc clusters on every other segment of a random cut of [0, M) (so some rows are in
    no cluster), each with up to max_ranges random column ranges in random order."""
    cuts = np.sort(r.choice(np.arange(1, M), size=2 * nc, replace=False))
    edges = np.concatenate([[0], cuts, [M]])
    ranges_i = np.stack([edges[1:-1:2], edges[2::2]], 1)[:nc]
    slices, red = [], []
    for _ in range(nc):
        for _ in range(int(r.integers(0, max_ranges + 1))):
            a = int(r.integers(0, N))
            red.append([a, int(r.integers(a, N + 1))])
        slices.append(len(red))
    return ranges_i, np.array(slices, dtype=np.int64), np.array(red, dtype=np.int64).reshape(-1, 2)


CASES = [(1500, 2000, 3, 1, 0.7, 6, 4), (700, 900, 16, 3, 2.0, 4, 3), (300, 400, 50, 1, 3.0, 3, 2),
         (200, 300, 128, 2, 6.0, 2, 3), (2100, 500, 2, 1, 0.5, 1, 6)]


@pytest.mark.parametrize("kernel", KINDS)
@pytest.mark.parametrize("M,N,D,E,sigma,nc,nr", CASES)
def test_ranges_random(orc, kernel, M, N, D, E, sigma, nc, nr):
    r = np.random.Generator(np.random.PCG64(M + N + D + len(kernel)))
    x = r.standard_normal((M, D)).astype(np.float32)
    y = r.standard_normal((N, D)).astype(np.float32)
    b = r.standard_normal((N, E)).astype(np.float32)
    ri, si, rj = _tables(r, M, N, nc, nr)
    xt, yt, bt = _t(x, y, b)
    a = kr.kernel_reduce_ranges(xt, yt, bt, sigma, "sum", ri, si, rj, kernel=kernel)
    a_ref, S_ref = orc.kernel_ranges(x, y, b, sigma, kernel, "sum", ri, si, rj)
    check_sum(_np(a), a_ref, S_ref, f"ranges sum {kernel}")
    for red in ("max", "min"):
        idx, val = kr.kernel_reduce_ranges(xt, yt, bt, sigma, red, ri, si, rj, want_index=True, kernel=kernel)
        v_ref, i_ref, s_ref = orc.kernel_ranges(x, y, b, sigma, kernel, red, ri, si, rj)
        check_maxmin(_np(val), _np(idx), x, y, b, sigma, kernel, v_ref, i_ref, s_ref, f"ranges {red} {kernel}")


def test_ranges_ties_lowest_index_out_of_order(orc):
    """Every point of y is one of 40 distinct points, repeated: duplicates have bitwise
    equal values, so each extreme is attained by a whole group of indices.  With the
    ranges listed from the top of [0, N) down, the lowest index must still win."""
    r = np.random.Generator(np.random.PCG64(41))
    x = r.standard_normal((600, 3)).astype(np.float32)
    y = r.standard_normal((40, 3)).astype(np.float32)[r.integers(0, 40, size=2000)]
    b = np.ones((2000, 1), np.float32)
    ri = np.array([[0, 250], [250, 600]])
    si = np.array([3, 5])
    rj = np.array([[1500, 2000], [700, 1500], [0, 700], [1000, 2000], [0, 1000]])
    for kernel in KINDS:
        for red in ("max", "min"):
            idx, _ = kr.kernel_reduce_ranges(*_t(x, y, b), 0.8, red, ri, si, rj, want_index=True, kernel=kernel)
            _, i_ref, _ = orc.kernel_ranges(x, y, b, 0.8, kernel, red, ri, si, rj)
            assert np.array_equal(_np(idx), i_ref), (kernel, red)


def test_ranges_truncated_product_on_sorted_points(orc):
    """The pages' use: points sorted into spatial clusters (here slabs along the first
    coordinate), each cluster of x reducing over its own and the neighbouring clusters
    of y.  Also: the dense cover (one cluster, one range) equals kernel_reduce."""
    r = np.random.Generator(np.random.PCG64(42))
    M, N, C = 4000, 6000, 10
    x = r.standard_normal((M, 3)).astype(np.float32)
    y = r.standard_normal((N, 3)).astype(np.float32)
    x = x[np.argsort(x[:, 0], kind="stable")]
    y = y[np.argsort(y[:, 0], kind="stable")]
    b = r.standard_normal((N, 1)).astype(np.float32)
    ex = np.linspace(0, M, C + 1).astype(np.int64)
    ey = np.linspace(0, N, C + 1).astype(np.int64)
    ri = np.stack([ex[:-1], ex[1:]], 1)
    rj = np.array([[ey[max(c - 1, 0)], ey[min(c + 2, C)]] for c in range(C)])
    si = np.arange(1, C + 1)
    xt, yt, bt = _t(x, y, b)
    a = kr.kernel_reduce_ranges(xt, yt, bt, 0.3, "sum", ri, si, rj)
    a_ref, S_ref = orc.kernel_ranges(x, y, b, 0.3, "gaussian", "sum", ri, si, rj)
    check_sum(_np(a), a_ref, S_ref, "truncated product")
    full = kr.kernel_reduce_ranges(xt, yt, bt, 0.3, "sum", [[0, M]], [1], [[0, N]])
    dense = kr.kernel_reduce(xt, yt, bt, 0.3, "sum")
    a_ref, S_ref = orc.gauss_sum(x, y, b, 0.3)
    check_sum(_np(full), a_ref, S_ref, "dense cover")
    check_sum(_np(dense), a_ref, S_ref, "dense")


def test_ranges_host_buffers_and_uncovered(orc):
    r = np.random.Generator(np.random.PCG64(43))
    x = r.standard_normal((300, 4)).astype(np.float32)
    y = r.standard_normal((500, 4)).astype(np.float32)
    b = r.standard_normal((500, 2)).astype(np.float32)
    ri, si, rj = np.array([[100, 200]]), np.array([1]), np.array([[0, 250]])
    host = kr.kernel_reduce_ranges(*(torch.from_numpy(a) for a in (x, y, b)), 1.0, "sum", ri, si, rj).numpy()
    dev = _np(kr.kernel_reduce_ranges(*_t(x, y, b), 1.0, "sum", ri, si, rj))
    assert np.array_equal(host, dev)
    assert (dev[:100] == 0).all() and (dev[200:] == 0).all() and (dev[100:200] != 0).any()
    idx, val = kr.kernel_reduce_ranges(*_t(x, y, b), 1.0, "min", ri, si, rj, want_index=True)
    assert (_np(idx)[:100] == -1).all() and np.isposinf(_np(val)[200:]).all()

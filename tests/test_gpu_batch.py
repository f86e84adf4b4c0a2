"""Batch dimension (kr_options.batch): B independent problems in one call, each
checked against the fp64 oracle, and against the same problem run alone with the same
forced split (which must give bit-identical results: a problem's arithmetic does not
depend on its neighbours in the batch)."""
import numpy as np
import pytest

import symbolic_matrix_reductions_gb300 as kr

from parity import check_grad, check_knn, check_lse, check_maxmin, check_sum

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


@pytest.fixture(scope="module")
def orc():
    import oracle
    return oracle.load()


def _np(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def _batch(seed, B, M, N, D, E):
    r = np.random.Generator(np.random.PCG64(seed))
    f = lambda *s: r.standard_normal(s).astype(np.float32)
    # each problem gets its own offset so that a mixed-up batch index shows
    off = np.arange(B, dtype=np.float32)[:, None, None] * 0.37
    return f(B, M, D) + off, f(B, N, D) + off, f(B, N, E), f(B, M, E)


def _t(*arrs):
    return [torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in arrs]


SHAPES = [(3, 700, 1100, 3, 1, 0.8), (4, 130, 257, 16, 2, 2.0), (2, 40, 90, 50, 1, 3.0), (5, 1, 1, 2, 3, 1.0),
          (2, 64, 300, 128, 4, 6.0)]


@pytest.mark.parametrize("B,M,N,D,E,sigma", SHAPES)
def test_batched_reductions_match_oracle(orc, B, M, N, D, E, sigma):
    x, y, b, g = _batch(B * 1000 + M + D, B, M, N, D, E)
    xt, yt, bt, gt = _t(x, y, b, g)
    a = _np(kr.kernel_reduce(xt, yt, bt, sigma, "sum"))
    L = _np(kr.kernel_reduce(xt, yt, bt, sigma, "lse"))
    gx = _np(kr.kernel_reduce_grad_x(xt, yt, bt, gt, sigma))
    gy = _np(kr.kernel_reduce_grad_y(xt, yt, bt, gt, sigma))
    gb = _np(kr.kernel_reduce_grad_b(xt, yt, gt, sigma))
    ac = _np(kr.kernel_reduce(xt, yt, bt, sigma, "sum", kernel="cauchy"))
    im, vm = (_np(t) for t in kr.kernel_reduce_arg(xt, yt, bt, sigma, "min", kernel="laplace"))
    K = min(5, N)
    ik, dk = (_np(t) for t in kr.kernel_knn(xt, yt, K))
    assert a.shape == (B, M, E) and gy.shape == (B, N, D) and ik.shape == (B, M, K)
    for p in range(B):
        w = f"problem {p} of {B}"
        ref, S = orc.gauss_sum(x[p], y[p], b[p], sigma)
        check_sum(a[p], ref, S, w)
        check_lse(L[p], orc.gauss_lse(x[p], y[p], b[p], sigma), w)
        ref, G = orc.gauss_grad_x(x[p], y[p], b[p], g[p], sigma)
        check_grad(gx[p], ref, G, w)
        ref, G = orc.gauss_grad_y(x[p], y[p], b[p], g[p], sigma)
        check_grad(gy[p], ref, G, w)
        ref, S = orc.gauss_grad_b(x[p], y[p], g[p], sigma)
        check_sum(gb[p], ref, S, w)
        ref, S = orc.kernel_sum(x[p], y[p], b[p], sigma, "cauchy")
        check_sum(ac[p], ref, S, w)
        v, i, sec = orc.kernel_maxmin(x[p], y[p], b[p], sigma, "laplace", "min")
        check_maxmin(vm[p], im[p], x[p], y[p], b[p], sigma, "laplace", v, i, sec, w)
        i_ref, d_ref, n_ref = orc.knn(x[p], y[p], K)
        check_knn(ik[p], dk[p], x[p], y[p], i_ref, d_ref, n_ref, w)


@pytest.mark.parametrize("split", [1, 3])
def test_batched_equals_single_problem(split):
    """Same forced split: a batched call and B single calls give bit-identical results."""
    B, M, N, D, E = 3, 600, 1500, 3, 2
    x, y, b, g = _batch(77, B, M, N, D, E)
    xt, yt, bt, gt = _t(x, y, b, g)
    outs = {
        "sum": lambda X, Y, Bv, G: kr.kernel_reduce(X, Y, Bv, 0.7, "sum", split=split),
        "lse": lambda X, Y, Bv, G: kr.kernel_reduce(X, Y, Bv, 0.7, "lse", split=split),
        "gx": lambda X, Y, Bv, G: kr.kernel_reduce_grad_x(X, Y, Bv, G, 0.7, split=split),
        "max": lambda X, Y, Bv, G: kr.kernel_reduce_arg(X, Y, Bv, 0.7, "max", split=split)[0],
        "knn": lambda X, Y, Bv, G: kr.kernel_knn(X, Y, 7, split=split)[0],
    }
    for name, fn in outs.items():
        batched = _np(fn(xt, yt, bt, gt))
        for p in range(B):
            single = _np(fn(xt[p].contiguous(), yt[p].contiguous(), bt[p].contiguous(), gt[p].contiguous()))
            assert np.array_equal(batched[p], single), (name, p)


def test_batched_autograd(orc):
    B, M, N, D = 2, 200, 300, 3
    x, y, b, _ = _batch(5, B, M, N, D, 1)
    xt, yt, bt = (t.requires_grad_(True) for t in _t(x, y, b))
    a = kr.GaussianSum.apply(xt, yt, bt, 0.9)
    gx, gy, gb = torch.autograd.grad((a ** 2).sum(), [xt, yt, bt])
    an = _np(a.detach())
    for p in range(B):
        ref, G = orc.gauss_grad_x(x[p], y[p], b[p], 2 * an[p], 0.9)
        check_grad(_np(gx)[p], ref, G, f"autograd x {p}")
        ref, G = orc.gauss_grad_y(x[p], y[p], b[p], 2 * an[p], 0.9)
        check_grad(_np(gy)[p], ref, G, f"autograd y {p}")
        ref, S = orc.gauss_grad_b(x[p], y[p], 2 * an[p], 0.9)
        check_sum(_np(gb)[p], ref, S, f"autograd b {p}")


def test_batched_host_buffers_and_empty(orc):
    x, y, b, _ = _batch(6, 3, 100, 200, 4, 2)
    host = kr.kernel_reduce(*(torch.from_numpy(a) for a in (x, y, b)), 1.0, "sum").numpy()
    dev = _np(kr.kernel_reduce(*_t(x, y, b), 1.0, "sum"))
    assert np.array_equal(host, dev)
    # N = 0 in every problem
    xt = _t(x)[0]
    e = torch.empty((3, 0, 4), device=DEV)
    eb = torch.empty((3, 0, 2), device=DEV)
    assert (_np(kr.kernel_reduce(xt, e, eb, 1.0, "sum")) == 0).all()
    assert np.isneginf(_np(kr.kernel_reduce(xt, e, eb, 1.0, "lse"))).all()
